// common.cuh -- device helpers shared by libmoe's kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// Device error codes recorded in the workspace error word.
constexpr int kDevErrBadExpert = 1;

// Bytes of a workspace's control region (its header and the row-tile counters), the same for
// every layer shape and token count (api.cu).
size_t workspace_control_bytes();

constexpr int kRouterPartials = 256;   // partial sums of the router's canonical order
constexpr int kMaxK = 32;              // top-k fits one warp
constexpr int kMaxE = 1024;
constexpr int kMaxDecodeCtas = 256;   // CTAs of the one-kernel decode layer at most (one per SM)
// The one-kernel layer's grid-barrier wait limit in ns (int64) sits at 32-bit word 4 past its
// barrier counters in the workspace header; zero means the default of one second.
constexpr int kWaitLimitWord = 4;

// Pointers into one layer workspace (see layout_for in api.cu).  The control words
// (err, route_ctr, the one-kernel layer's counters, row_ctr) sit at fixed offsets in the
// first workspace_control_bytes() bytes; they must be zero before a call, and the kernels
// leave the counters zero again when they finish.
struct Workspace {
    int32_t* err;          // [1] sticky first error
    int32_t* route_ctr;    // [1] CTAs of the routing kernel that have finished their logits
    int32_t* row_ctr;      // [d/32] down CTAs finished per row tile (fused combine); room for the largest d
    int32_t* n_active;     // [1] number of experts with at least one pair
    float* logits;         // [T][E]
    float* rpart;          // [T][E][32] router partial sums by residue class (fused decode routing)
    int32_t* idx;          // [T][k]
    float* w;              // [T][k]
    int32_t* offsets;      // [E+1]
    int32_t* perm;         // [P] sorted row -> pair
    int32_t* pos;          // [P] pair -> sorted row
    int32_t* act_e;        // [min(E,P)] expert id of each active slot, increasing
    int4* slot_info;       // [min(E,P)] per slot: expert, first sorted row, pair count (0 = idle slot),
                           //   and the tokens of its first four rows packed 8 bits each (-1: read perm)
    int32_t* chunk_cnt;    // [nchunk][E] pairs of each expert per chunk (large-T permute)
    int32_t* local_rank;   // [P] rank of a pair among its expert's pairs in its chunk
    uint32_t* gmask;       // [min(E,P)][ceil(f/16/32)] active 16-neuron groups per slot
    float* h;              // [P][f] activations, sorted rows
    float* y;              // [P][d] down projections, sorted rows
    uint16_t* xs_hi;       // [P][d] f16 x in sorted-row order (tensor-core path), hi part
    uint16_t* xs_lo;       // [P][d] ... lo part (fp32 inputs)
    uint16_t* h_hi;        // [P][f] f16 hi part of h (tensor-core path)
    uint16_t* h_lo;        // [P][f] f16 lo part of h
};

// Arguments of the expert kernels (gate.up, down) of one layer call.
struct ExpertArgs {
    const void* x;
    int xt;
    int d, f, k, rows_gu;
    int tt_gu, tt_dn;            // tokens per shared-memory tile
    int gu_wpt;                  // gate.up: warps that share one tile's K panels (8, 4, 2 or 1)
    int gwords;                  // 32-bit words of group mask per slot
    int T;                       // tokens
    int P;                       // pairs T*k
    int fuse_combine;            // the down kernel's last CTA per row tile also combines
    int prefetch_down;           // gate.up CTAs prefetch the routed experts' down weights into L2
    int nv_split;                // NVFP4 down, fused combine: CTAs per (row tile, slot), each a share of the groups
    int nv_mma;                  // NVFP4 down on the tensor cores (two or more tokens; tt_dn = 8, 16 or 32)
    float* out;                  // [T][d] layer output (fused combine)
    const uint8_t* w_gu;
    int64_t gu_bytes;            // bytes of one expert's gate/up matrix
    const uint8_t* w_dn;
    int64_t dn_bytes;
    const uint8_t* pf;           // bytes to pull into L2 during the gate.up kernel (a hint), or null
    int64_t pf_bytes;
    const float* gu_ts;          // NVFP4 tensor scales [E] (or null)
    const float* dn_ts;
    Workspace ws;
};

// Arguments of the one-kernel decode layer (decode.cu): one token, Q8_0 SwiGLU or NVFP4 ReLU^2
// experts, one layer or a stack of layers of the same shape (the next layer's input is the
// RMS-normalised output of the previous one), routed in the kernel or (one layer) by the
// caller's idx / w.  The kernel's own control words and partial sums sit in the layer
// workspace too.
constexpr int kMaxStackLayers = 64;

struct DecodeLayerPtrs {
    const float* W;              // router [d][E]
    const uint8_t* w_gu;         // gate/up matrices of the E experts (Q8_0 device layout, or NVFP4 panels)
    const uint8_t* w_dn;         // down matrices (Q8_0 device layout, or NVFP4 neuron-contiguous)
    const uint8_t* pf;           // L2 hint (the next layer's router weights), or null
    int64_t pf_bytes;
    const float* gu_ts;          // NVFP4 tensor scales [E] of the gate/up and down matrices
    const float* dn_ts;
};

struct DecodeArgs {
    const void* x;               // the first layer's input [d]
    int xt;
    int d, f, E, k;
    int epc;                     // router experts per routing CTA (E / epc CTAs compute logits)
    int prefetch_down;           // the routed experts' down matrices are pulled into L2 during gate.up
    int warps_g, warps_d;        // warps that share the gate.up / down panel ranges
    int cov_g, cov_d;            // partial records per item at most (CTAs / warps that can share one item)
    int cta_items;               // gate.up items one CTA's range touches at most
    int cta_items_d;             // NVFP4: down items (slot, 256-row tile) one CTA's range touches at most
    int off_c, off_p;            // dynamic shared memory offsets of x f16 and the gate.up partials (bytes)
    int64_t gu_bytes, dn_bytes;  // bytes of one expert's gate/up and down matrices
    int n_layers;                // 1: moe_layer_forward; more: moe_stack_forward
    float eps;                   // RMS-norm between stacked layers
    float* out;                  // [n_layers][d] every layer's output
    uint16_t* x_next;            // [n_layers][d] bf16 RMS-normalised outputs (stacks; may be null)
    int32_t* idx_out;            // [n_layers][k] routing of each layer (stacks; may be null)
    float* w_out;                // [n_layers][k]
    Workspace ws;
    int32_t* bar;                // [2] grid-barrier arrivals, CTAs finished (zero between calls);
                                 //   bar[kWaitLimitWord..+1]: the barrier wait limit (int64 ns, 0 = 1 s)
    int32_t* sel;                // [k] experts selected by rank (more than 256 experts)
    float* selv;                 // [k] their logits
    float* grec;                 // [k * f/16][cov_g][32] gate.up partial sums per item and contributor
    float* drec;                 // [k * d/32][cov_d][32] (Q8_0) or [k * d/256][cov_d][256] (NVFP4) down
                                 //   partial sums per item and contributor
    DecodeLayerPtrs lp[kMaxStackLayers];
    // last, so that the offsets of the fields above (and the routed kernels' code) stay as they were
    const int32_t* idx_in;       // supplied routing [k] and weights [k] (one layer), or null: routed here
    const float* w_in;
    int act_q;                   // 1: the experts read Q8_0-coded x and h (the AQ instantiation; host-side dispatch)
};

// Programmatic dependent launch: wait for the preceding kernel's memory, and allow the
// next kernel to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialization allowed (the kernel calls pdl_wait()
// before touching global memory, so overlap with the previous kernel is safe).
template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

constexpr int kNoPackedTokens = -1;

// Token of sorted row r0 + i of a slot, from the packed field when present.
__device__ __forceinline__ int slot_token(const int4& si, int i, const int32_t* perm, int k) {
    if (si.w != kNoPackedTokens && i < 4) return (si.w >> (8 * i)) & 0xff;
    return perm[si.y + i] / k;
}

__device__ __forceinline__ void set_error(int32_t* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// x row element as fp32 (exact for bf16).
__device__ __forceinline__ float load_x(const void* x, int xt, int64_t off) {
    if (xt == MOE_F32) return static_cast<const float*>(x)[off];
    return bf16_bits_to_f32(static_cast<const uint16_t*>(x)[off]);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Signed int8 byte b of a 32-bit word as float, exact.
__device__ __forceinline__ float s8_to_f32(uint32_t word, int b) {
    return static_cast<float>(static_cast<int8_t>((word >> (8 * b)) & 0xffu));
}

// Two E2M1 codes (one byte, low nibble first) -> two floats, exact.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
    __half2 hh = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(hh);   // .x = low half = the low nibble's code
}

// One E4M3 byte -> float, exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    uint32_t h2;
    uint16_t in = static_cast<uint16_t>(byte & 0xffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h2 & 0xffffu)));
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// The Q8_0 activation coder for one value of a block of 32 whose largest magnitude is amax:
// d = amax / 127, the code round(x * (1 / d)) (both correctly rounded, as the weight packer),
// and the value the code stands for, q * fp16(d), which is exact in fp32.
__device__ __forceinline__ float q8_0_coded_value(float x, float amax) {
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    const int q = static_cast<int>(roundf(__fmul_rn(x, id)));
    return static_cast<float>(q) * __half2float(__float2half_rn(d));
}

// Two fp32 fused multiply-adds in one instruction, each half rounded as fmaf:
// acc.lo = fma(a.lo, b.lo, acc.lo), acc.hi = fma(a.hi, b.hi, acc.hi).
__device__ __forceinline__ void fma_f32x2(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// Two fp32 additions in one instruction, each half rounded as an fp32 add.
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

}  // namespace moe
