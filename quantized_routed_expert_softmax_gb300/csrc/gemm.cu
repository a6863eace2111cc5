// gemm.cu -- expert kernels for many tokens per expert: grouped GEMMs on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// gate.up + activation and the down projection of the routed layer ("Running Gemma 4 26B
// at 5 tokens/s on a 13-year-old Xeon", section "A three-step fix" / "Runtime graph
// fallback": per-expert matmuls over the gate-first/up-second [n_embd, 2*n_ff, n_experts]
// tensor; "Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU", "bytes per token":
// the gateless ReLU^2 latent experts), for batches where each expert sees many tokens.
//
// Swap-AB: D[128 weight rows][N tokens] = W_e[rows][K] * B^T, so the weight rows fill the
// MMA's M = 128 and the expert's tokens fill N (16..256).  B is an f16 "plane" of
// activations in sorted-row order ([P][K]; written by gather_x_f16_kernel for gate.up and by
// the gate.up epilogue for down), so a token tile is a plain 2-D box that TMA copies straight
// into the 128-byte-swizzled K-major layout the tensor core reads.  fp32 activations (fp32
// inputs, and always the hidden activations h) come as two planes hi + lo.
//
// A persistent grid walks a device-built list of (expert slot, token tile, row tile) work
// items.  The warps of a CTA have fixed roles, linked by mbarriers:
//   warp 0       weight producer: 1-D bulk copies of each K step's raw Q8_0 / NVFP4 bytes
//                into a ring of kRawSlots slots (several K steps of HBM reads in flight);
//   warp 1       activation producer: TMA 2-D loads of the token tile's B planes;
//   warp 2       MMA issuer (one thread): per K step of 64, four K = 16 slices of
//                tcgen05.mma (A.hi*B.hi, A.lo*B.hi for Q8_0, A.hi*B.lo for two planes; the
//                lo*lo term is below fp32 rounding), committed to the stage's "empty"
//                barrier, and at the end of an item to the accumulator's "full" barrier;
//   warps 4..7   epilogue: tensor memory -> registers (lane quadrant = warp % 4), the
//                activation (SwiGLU pairs gate row i and up row i on accumulator lanes 2i
//                and 2i+1, one shuffle), stores; two accumulators alternate, so the
//                epilogue of one item overlaps the main loop of the next;
//   warps 8..15  dequantisers: raw slot -> f16 A tiles.  NVFP4 weights e2m1 * e4m3 are
//                exact in f16.  A Q8_0 weight q * d needs up to 18 significant bits, so it
//                is split into hi = f16(q * d) and lo = fma(q, d, -hi), the exact residual
//                rounded once.
// Every wait on an mbarrier is bounded (about a second); on timeout the kernel records MOE
// device error 2, waits (bounded) for its copies and MMAs in flight, releases its tensor
// memory and returns.
#include <cuda.h>   // CUtensorMap and its enums; the encoder is looked up in the driver at run time
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moe {

constexpr int kDevErrTimeout = 2;
constexpr int kDevErrF16Range = 3;
constexpr long long kWaitLimitNs = 1000000000ll;

constexpr int kGemmThreads = 512;
constexpr int kTileM = 128;
constexpr int kStepK = 64;                          // one 128-byte swizzle row of f16
constexpr int kBRows = 256;                         // B rows per stage: token tile x planes
constexpr int kBoxRows = 32;                        // rows per TMA box
constexpr int kRawSlots = 8;
constexpr int kStages = 2;
constexpr int kRawSlot = 9216;                      // >= 8704 (Q8_0: 2 panels x (4096 + 256))
constexpr int kATile = kTileM * kStepK * 2;         // 16 KB
constexpr int kBTile = kBRows * kStepK * 2;         // 32 KB
constexpr int kStageBytes = 2 * kATile + kBTile;    // A hi, A lo, B planes
constexpr size_t kGemmSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes +
                             static_cast<size_t>(kRawSlots) * kRawSlot;
constexpr int kWarpLoadA = 0, kWarpLoadB = 1, kWarpMma = 2, kWarpEpi0 = 4, kWarpConv0 = 8;
constexpr int kConvWarps = 8, kConvThreads = kConvWarps * 32;

// ------------------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t s_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ long long global_ns() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(s_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(s_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(s_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for completion number n (0-based) of a barrier's phases, for at most kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t n) {
    const uint32_t parity = n & 1u;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(s_addr(bar))
                 : "memory");
}

// TMA 2-D tile load (coordinates: x = column, y = row), completion on `bar`.
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(s_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, rows of 128 bytes, 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1 (tcgen05).
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused by this layout)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                 // version
    d |= static_cast<uint64_t>(2) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B, both K-major, M = 128.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kTileM >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(s_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// f16 hi + lo of an fp32 value (hi + lo carries about 22 significant bits).
__device__ __forceinline__ void split_f16(float v, __half* hi, __half* lo) {
    *hi = __float2half_rn(v);
    *lo = __float2half_rn(v - __half2float(*hi));
}

// ------------------------------------------------------------------------------ work items
enum GemmKind { kGateUp = 0, kDown = 1 };

struct GemmArgs {
    CUtensorMap tb[2];   // B planes, f16 [P][K] (hi, lo), boxes of 64 columns x kBoxRows rows
    ExpertArgs a;
    int kind;            // GemmKind
    int fmt;             // MOE_W_Q8_0 / MOE_W_NVFP4
    int act;             // MOE_ACT_* (gate.up)
    int slot_cap;
    int planes;          // 1 or 2
    int nt_max;          // token tile: kBRows / planes
};

struct Item {
    int e;               // expert
    int r_first;         // first sorted row of the token tile
    int nt;              // tokens in the tile (1..nt_max)
    int mtile;           // row tile
};

__device__ __forceinline__ Item decode_item(const GemmArgs& g, const int* tile_prefix, int mtiles, int item) {
    int lo = 0, hi = g.slot_cap - 1;
    while (lo < hi) {   // last slot whose first item is <= item
        const int mid = (lo + hi + 1) >> 1;
        if (tile_prefix[mid] <= item) lo = mid;
        else hi = mid - 1;
    }
    const int4 si = __ldcg(g.a.ws.slot_info + lo);
    const int local = item - tile_prefix[lo];
    const int ntile = local / mtiles;
    Item it;
    it.e = si.x;
    it.mtile = local - ntile * mtiles;
    it.r_first = si.y + ntile * g.nt_max;
    it.nt = min(g.nt_max, si.z - ntile * g.nt_max);
    return it;
}

// Raw bytes of one K step of the weights.
__device__ __forceinline__ uint32_t raw_step_bytes(const GemmArgs& g) {
    return (g.fmt == MOE_W_Q8_0) ? 2u * (4096u + 256u) : 4096u + 512u;
}

// The weight producer's copies of K step ks for row tile `mtile` of expert matrix W
// (lane-strided).  Raw slot layout: Q8_0 two panels of 32 columns, each [128 rows][32 codes]
// then [128][2-byte scale] at 4608-byte spacing; NVFP4 one panel of 64 columns, [128][32
// code bytes] then [128][4 scale bytes]; NVFP4 down (neuron layout) four 16-neuron groups
// at 1152-byte spacing, each [16 neurons][64 bytes = 128 rows' nibbles] then [128 scales].
// SwiGLU gate.up tiles stage gate rows in rows 0..63 and the same neurons' up rows in 64..127.
__device__ __forceinline__ void issue_weights(const GemmArgs& g, uint32_t slot_addr, const uint8_t* W, int rows_w,
                                              int mtile, int ks, uint64_t* bar, int lane) {
    const ExpertArgs& a = g.a;
    const bool swiglu = (g.kind == kGateUp && g.act == MOE_ACT_SWIGLU);
    if (g.kind == kDown && g.fmt == MOE_W_NVFP4) {
        const int64_t rec = 16 * static_cast<int64_t>(a.d / 2) + a.d;   // one 16-neuron group record
        const int row0 = mtile * kTileM;
        for (int c = lane; c < 4 * 17; c += 32) {
            const int grp = c / 17, n = c % 17;
            const uint8_t* base = W + (static_cast<int64_t>(ks) * 4 + grp) * rec;
            if (n < 16)
                bulk_g2s(slot_addr + grp * 1152 + n * 64, base + static_cast<int64_t>(n) * (a.d / 2) + row0 / 2, 64, bar);
            else
                bulk_g2s(slot_addr + grp * 1152 + 1024, base + 16 * static_cast<int64_t>(a.d / 2) + row0, 128, bar);
        }
        return;
    }
    const bool q8 = (g.fmt == MOE_W_Q8_0);
    const int npanel = q8 ? 2 : 1;
    const int scb = q8 ? 2 : 4;                                  // scale bytes per row per panel
    const int64_t pbytes = static_cast<int64_t>(rows_w) * (q8 ? 34 : 36);
    const int runs = swiglu ? 2 : 1;                             // row runs per panel
    const int run_rows = kTileM / runs;
    const int ncopies = npanel * runs * 2;
    for (int c = lane; c < ncopies; c += 32) {
        const int p = c / (runs * 2), rem = c % (runs * 2);
        const int run = rem >> 1, is_scale = rem & 1;
        const int src_row = swiglu ? (run == 0 ? mtile * 64 : a.f + mtile * 64) : mtile * kTileM;
        const uint8_t* P = W + (static_cast<int64_t>(ks) * npanel + p) * pbytes;
        const uint32_t dst = slot_addr + p * 4608;
        if (!is_scale)
            bulk_g2s(dst + run * run_rows * 32, P + static_cast<int64_t>(src_row) * 32, run_rows * 32, bar);
        else
            bulk_g2s(dst + 4096 + run * run_rows * scb, P + static_cast<int64_t>(rows_w) * 32 + src_row * scb,
                     run_rows * scb, bar);
    }
}

// Dequantise one K step from a raw slot into the A hi (and, for Q8_0, lo) tiles.
__device__ __forceinline__ void dequant_step(const GemmArgs& g, const unsigned char* raw, unsigned char* ta,
                                             unsigned char* tal, int ct) {
    const bool swiglu = (g.kind == kGateUp && g.act == MOE_ACT_SWIGLU);
#pragma unroll
    for (int i = 0; i < (kTileM * 4) / kConvThreads; ++i) {
        const int u = ct + i * kConvThreads;
        const int r = u >> 2, c16 = u & 3;              // tile row, 16-column chunk
        const int sr = swiglu ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;   // staged row
        uint32_t h[8];
        if (g.fmt == MOE_W_Q8_0) {
            const int p = c16 >> 1, hh = c16 & 1;       // panel of 32 columns, half
            const unsigned char* pan = raw + p * 4608;
            const uint4 q = *reinterpret_cast<const uint4*>(pan + sr * 32 + hh * 16);
            const unsigned short sbits = *reinterpret_cast<const unsigned short*>(pan + 4096 + sr * 2);
            const __half2 s2 = __halves2half2(__ushort_as_half(sbits), __ushort_as_half(sbits));
            const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
            uint32_t hl[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // int8 codes -> exact f16: bytes XOR 0x80 placed under exponent 0x64 give
                // 1024 + 128 + q; subtracting 1152 (0x6480) leaves q
                const uint32_t u8 = w4[j] ^ 0x80808080u;
                const uint32_t b01 = __byte_perm(u8, 0x64646464u, 0x4140);
                const uint32_t b23 = __byte_perm(u8, 0x64646464u, 0x4342);
                const __half2 q01 = __hsub2(*reinterpret_cast<const __half2*>(&b01), off);
                const __half2 q23 = __hsub2(*reinterpret_cast<const __half2*>(&b23), off);
                const __half2 v01 = __hmul2(q01, s2), v23 = __hmul2(q23, s2);
                const __half2 l01 = __hfma2(q01, s2, __hneg2(v01)), l23 = __hfma2(q23, s2, __hneg2(v23));
                h[2 * j] = *reinterpret_cast<const uint32_t*>(&v01);
                h[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&v23);
                hl[2 * j] = *reinterpret_cast<const uint32_t*>(&l01);
                hl[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&l23);
            }
            *reinterpret_cast<uint4*>(tal + swz(r, 2 * c16)) = make_uint4(hl[0], hl[1], hl[2], hl[3]);
            *reinterpret_cast<uint4*>(tal + swz(r, 2 * c16 + 1)) = make_uint4(hl[4], hl[5], hl[6], hl[7]);
        } else if (g.kind == kDown) {
            // NVFP4 neuron layout: columns 16*c16 .. +15 are group c16; row sr is nibble
            // (sr & 1) of byte sr/2 in each neuron's run
            const unsigned char* gb = raw + c16 * 1152;
            uint32_t s16;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(static_cast<uint16_t>(gb[1024 + sr])));
            const __half sh = __ushort_as_half(static_cast<unsigned short>(s16 & 0xffffu));
            const __half2 s2 = __halves2half2(sh, sh);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t b0 = gb[(2 * j) * 64 + (sr >> 1)];
                const uint32_t b1 = gb[(2 * j + 1) * 64 + (sr >> 1)];
                const uint32_t n0 = (sr & 1) ? (b0 >> 4) : (b0 & 0xfu);
                const uint32_t n1 = (sr & 1) ? (b1 >> 4) : (b1 & 0xfu);
                uint32_t h2;
                asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(n0 | (n1 << 4)));
                const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), s2);
                h[j] = *reinterpret_cast<const uint32_t*>(&v);
            }
        } else {
            // NVFP4 panel of 64 columns: 32 code bytes, 4 scale bytes per row
            const uint2 cw = *reinterpret_cast<const uint2*>(raw + sr * 32 + c16 * 8);
            uint32_t s16;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(static_cast<uint16_t>(raw[4096 + sr * 4 + c16])));
            const __half sh = __ushort_as_half(static_cast<unsigned short>(s16 & 0xffffu));
            const __half2 s2 = __halves2half2(sh, sh);
            const uint32_t w2[2] = {cw.x, cw.y};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t h2;
                const uint32_t byte = (w2[j >> 2] >> (8 * (j & 3))) & 0xffu;
                asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
                const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), s2);
                h[j] = *reinterpret_cast<const uint32_t*>(&v);
            }
        }
        *reinterpret_cast<uint4*>(ta + swz(r, 2 * c16)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(ta + swz(r, 2 * c16 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

// ------------------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kGemmThreads, 1) expert_gemm_kernel(const __grid_constant__ GemmArgs g) {
    pdl_wait();
    const ExpertArgs& a = g.a;
    extern __shared__ __align__(16) unsigned char dsm_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* stages = base;                               // kStages x (A hi, A lo, B)
    unsigned char* raws = base + kStages * kStageBytes;         // kRawSlots x kRawSlot
    __shared__ uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];
    __shared__ uint64_t a_full[kStages], b_full[kStages], st_empty[kStages];
    __shared__ uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t raw_issued[kRawSlots], b_issued[kStages], mma_commits[kStages];
    __shared__ uint32_t tmem_base;
    __shared__ int tile_prefix[kMaxE + 1];
    __shared__ int warp_tot[kGemmThreads / 32];
    __shared__ volatile int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t tmem_cols = static_cast<uint32_t>(2 * g.nt_max);   // two accumulators

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(&tmem_base)),
                     "r"(tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int s = 0; s < kRawSlots; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kConvWarps);
            raw_issued[s] = 0;
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&a_full[s], kConvWarps);
            mbar_init(&b_full[s], 1);
            mbar_init(&st_empty[s], 1);
            b_issued[s] = 0;
            mma_commits[s] = 0;
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_fail = 0;
    }
    // the work list: per slot, (token tiles) x (row tiles); exclusive prefix over the slots
    const int rows_out = (g.kind == kGateUp) ? a.rows_gu : a.d;
    const int mtiles = rows_out / kTileM;
    {
        const int per = (g.slot_cap + kGemmThreads - 1) / kGemmThreads;   // <= 2 (slot_cap <= 1024)
        const int s0 = tid * per;
        int cnts[2] = {0, 0};
        int local = 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (i < per && s0 + i < g.slot_cap) {
                const int c = __ldcg(&a.ws.slot_info[s0 + i].z);
                cnts[i] = ((c + g.nt_max - 1) / g.nt_max) * mtiles;
            }
            local += cnts[i];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int run = incl - local;
        for (int w = 0; w < warp; ++w) run += warp_tot[w];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (i < per && s0 + i < g.slot_cap) tile_prefix[s0 + i] = run;
            run += cnts[i];
        }
        if (tid == kGemmThreads - 1) tile_prefix[g.slot_cap] = run;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const int total = tile_prefix[g.slot_cap];
    const int ksteps = ((g.kind == kGateUp) ? a.d : a.f) / kStepK;
    const int rows_w = (g.kind == kGateUp) ? a.rows_gu : a.d;

    if (warp == kWarpLoadA) {
        // ---------------------------------------------------------------- weight producer
        const uint32_t bytes = raw_step_bytes(g);
        uint32_t gs = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            const Item it = decode_item(g, tile_prefix, mtiles, item);
            const uint8_t* W = (g.kind == kGateUp) ? a.w_gu + static_cast<int64_t>(it.e) * a.gu_bytes
                                                   : a.w_dn + static_cast<int64_t>(it.e) * a.dn_bytes;
            for (int ks = 0; ks < ksteps; ++ks, ++gs) {
                const int slot = gs % kRawSlots;
                const uint32_t use = gs / kRawSlots;
                bool w_ok = (use == 0) || mbar_wait(&raw_empty[slot], use - 1);
                w_ok = __all_sync(0xffffffffu, w_ok) && !s_fail;
                if (!w_ok) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&raw_full[slot], bytes);
                    raw_issued[slot] = use + 1;
                }
                __syncwarp();
                issue_weights(g, s_addr(raws + slot * kRawSlot), W, rows_w, it.mtile, ks, &raw_full[slot], lane);
            }
        }
        if (!ok && lane == 0) {
            s_fail = 1;
            atomicCAS(a.ws.err, 0, kDevErrTimeout);
        }
    } else if (warp == kWarpLoadB) {
        // ---------------------------------------------------------------- activation producer
        if (lane == 0) {
            uint32_t gs = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const Item it = decode_item(g, tile_prefix, mtiles, item);
                const int nbox = (it.nt + kBoxRows - 1) / kBoxRows;
                const uint32_t bytes = static_cast<uint32_t>(nbox * kBoxRows * 128 * g.planes);
                for (int ks = 0; ks < ksteps; ++ks, ++gs) {
                    const int st = gs % kStages;
                    const uint32_t use = gs / kStages;
                    if ((use > 0 && !mbar_wait(&st_empty[st], use - 1)) || s_fail) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&b_full[st], bytes);
                    b_issued[st] = use + 1;
                    const uint32_t bdst = s_addr(stages + st * kStageBytes + 2 * kATile);
                    for (int p = 0; p < g.planes; ++p)
                        for (int j = 0; j < nbox; ++j)
                            tma_2d(bdst + p * g.nt_max * 128 + j * kBoxRows * 128, &g.tb[p], ks * kStepK,
                                   it.r_first + j * kBoxRows, &b_full[st]);
                }
            }
            if (!ok) {
                s_fail = 1;
                atomicCAS(a.ws.err, 0, kDevErrTimeout);
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const bool alo = (g.fmt == MOE_W_Q8_0);
            uint32_t gs = 0, n_item = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++n_item) {
                const Item it = decode_item(g, tile_prefix, mtiles, item);
                const int n16 = (it.nt + 15) & ~15;
                const uint32_t idesc = idesc_f16(n16);
                const int buf = n_item & 1;
                const uint32_t ub = n_item >> 1;
                if ((ub > 0 && !mbar_wait(&acc_empty[buf], ub - 1)) || s_fail) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + static_cast<uint32_t>(buf * g.nt_max);
                for (int ks = 0; ks < ksteps; ++ks, ++gs) {
                    const int st = gs % kStages;
                    const uint32_t use = gs / kStages;
                    if (!mbar_wait(&a_full[st], use) || !mbar_wait(&b_full[st], use) || s_fail) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = s_addr(stages + st * kStageBytes);
                    const uint32_t sal = sa + kATile;
                    const uint32_t sb = sa + 2 * kATile;
                    const uint32_t sbl = sb + g.nt_max * 128;
#pragma unroll
                    for (int kk = 0; kk < kStepK / 16; ++kk) {
                        umma_f16(dt, sdesc_k128(sa + kk * 32), sdesc_k128(sb + kk * 32), idesc, (ks | kk) ? 1u : 0u);
                        if (alo) umma_f16(dt, sdesc_k128(sal + kk * 32), sdesc_k128(sb + kk * 32), idesc, 1u);
                        if (g.planes == 2) umma_f16(dt, sdesc_k128(sa + kk * 32), sdesc_k128(sbl + kk * 32), idesc, 1u);
                    }
                    umma_commit(&st_empty[st]);
                    mma_commits[st] = use + 1;
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);
            }
            if (!ok) {
                s_fail = 1;
                atomicCAS(a.ws.err, 0, kDevErrTimeout);
            }
        }
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;                 // accumulator lane = tile row
        const float* ts_arr = (g.kind == kGateUp) ? a.gu_ts : a.dn_ts;
        uint32_t n_item = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total; item += gridDim.x, ++n_item) {
            const Item it = decode_item(g, tile_prefix, mtiles, item);
            const int n16 = (it.nt + 15) & ~15;
            const int buf = n_item & 1;
            bool w_ok = mbar_wait(&acc_full[buf], n_item >> 1);
            w_ok = __all_sync(0xffffffffu, w_ok) && !s_fail;
            if (!w_ok) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float ts = (g.fmt == MOE_W_NVFP4) ? ts_arr[it.e] : 1.0f;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * g.nt_max);
            bool range_ok = true;
            for (int c0 = 0; c0 < n16; c0 += 16) {
                float v[16];
                tmem_ld16(tbase + static_cast<uint32_t>(c0), v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c0 + j;
                    const int64_t prow = static_cast<int64_t>(it.r_first + n);
                    const float z = v[j] * ts;
                    if (g.kind == kGateUp) {
                        float hv;
                        int64_t col;
                        bool store;
                        if (g.act == MOE_ACT_SWIGLU) {
                            const float u = __shfl_xor_sync(0xffffffffu, z, 1);   // odd lanes hold the up rows
                            hv = silu(z) * u;
                            col = it.mtile * 64 + (row >> 1);
                            store = !(lane & 1) && n < it.nt;
                        } else {
                            hv = z > 0.0f ? z * z : 0.0f;
                            col = it.mtile * kTileM + row;
                            store = n < it.nt;
                        }
                        if (store) {
                            const int64_t o = prow * a.f + col;
                            a.ws.h[o] = hv;
                            __half hh, hl;
                            split_f16(hv, &hh, &hl);
                            range_ok &= fabsf(hv) <= 65504.0f;
                            a.ws.h_hi[o] = __half_as_ushort(hh);
                            a.ws.h_lo[o] = __half_as_ushort(hl);
                        }
                    } else if (n < it.nt) {
                        a.ws.y[prow * a.d + it.mtile * kTileM + row] = z;
                    }
                }
            }
            if (!range_ok) atomicCAS(a.ws.err, 0, kDevErrF16Range);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (!ok && lane == 0) {
            s_fail = 1;
            atomicCAS(a.ws.err, 0, kDevErrTimeout);
        }
    } else if (warp >= kWarpConv0) {
        // ---------------------------------------------------------------- dequantisers
        const int ct = tid - kWarpConv0 * 32;
        int my_items = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) ++my_items;
        const uint32_t nsteps = static_cast<uint32_t>(my_items) * ksteps;
        bool ok = true;
        for (uint32_t gs = 0; gs < nsteps; ++gs) {
            const int slot = gs % kRawSlots;
            const int st = gs % kStages;
            const uint32_t use = gs / kStages;
            bool w_ok = mbar_wait(&raw_full[slot], gs / kRawSlots);
            w_ok = w_ok && (use == 0 || mbar_wait(&st_empty[st], use - 1));
            w_ok = __all_sync(0xffffffffu, w_ok) && !s_fail;
            if (!w_ok) {
                ok = false;
                break;
            }
            unsigned char* sa = stages + st * kStageBytes;
            dequant_step(g, raws + slot * kRawSlot, sa, sa + kATile, ct);
            proxy_fence_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a_full[st]);
                mbar_arrive(&raw_empty[slot]);
            }
        }
        if (!ok && lane == 0) {
            s_fail = 1;
            atomicCAS(a.ws.err, 0, kDevErrTimeout);
        }
    }

    // drain: every copy and MMA this CTA issued has landed before shared and tensor memory
    // are given back (immediate on the normal path; bounded after a timeout)
    __syncthreads();
    if (tid == 0) {
        bool ok = true;
        for (int s = 0; s < kRawSlots; ++s)
            if (raw_issued[s]) ok &= mbar_wait(&raw_full[s], raw_issued[s] - 1);
        for (int s = 0; s < kStages; ++s) {
            if (b_issued[s]) ok &= mbar_wait(&b_full[s], b_issued[s] - 1);
            if (mma_commits[s]) ok &= mbar_wait(&st_empty[s], mma_commits[s] - 1);
        }
        if (!ok) atomicCAS(a.ws.err, 0, kDevErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols));
}

// f16 B planes of the gate.up GEMM: x rows in sorted-row order (hi = f16(x); for fp32 x
// also lo = f16(x - hi)).  One thread per 8 elements, grid-stride.
__global__ void __launch_bounds__(256) gather_x_f16_kernel(const void* __restrict__ x, int xt, int d, int k,
                                                           int64_t P, const int32_t* __restrict__ perm,
                                                           uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                                                           int32_t* err) {
    pdl_wait();
    pdl_trigger();
    const int cpr = d / 8;
    const int64_t total = P * cpr;
    bool range_ok = true;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t p = i / cpr;
        const int c = static_cast<int>(i - p * cpr);
        const int64_t t = __ldg(perm + p) / k;
        float v[8];
        if (xt == MOE_F32) {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + t * d) + 2 * c;
            const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
            v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
            v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        } else {
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + t * d) + c);
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[2 * j] = __uint_as_float(bw[j] << 16);
                v[2 * j + 1] = __uint_as_float(bw[j] & 0xffff0000u);
            }
        }
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half h0, l0, h1, l1;
            split_f16(v[2 * j], &h0, &l0);
            split_f16(v[2 * j + 1], &h1, &l1);
            range_ok &= fabsf(v[2 * j]) <= 65504.0f && fabsf(v[2 * j + 1]) <= 65504.0f;
            hw[j] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
            lw[j] = static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
        }
        reinterpret_cast<uint4*>(hi + p * d)[c] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if (xt == MOE_F32) reinterpret_cast<uint4*>(lo + p * d)[c] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    if (!range_ok) atomicCAS(err, 0, kDevErrF16Range);
}

// ------------------------------------------------------------------------------ host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    static std::once_flag once;
    static cudaError_t status = cudaSuccess;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (status == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr)) status = cudaErrorNotSupported;
        if (status == cudaSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return status;
}

// Tensor map of an f16 plane [rows][cols] (row stride cols*2 bytes), boxes of 64 columns x
// kBoxRows rows, 128-byte swizzle; rows past the end read as zero.
cudaError_t plane_map(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t cols) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kStepK), static_cast<cuuint32_t>(kBoxRows)};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box,
                                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t configure_gemm_kernels() {
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(expert_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(expert_gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

size_t gemm_smem_bytes() { return kGemmSmem; }

cudaError_t launch_gather_x_f16(const ExpertArgs& a, int num_sms, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(a.P) * (a.d / 8);
    const int64_t want = (total + 255) / 256;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(num_sms) * 8)));
    return launch_pdl(gather_x_f16_kernel, dim3(grid), dim3(256), 0, s, a.x, a.xt, a.d, a.k,
                      static_cast<int64_t>(a.P), static_cast<const int32_t*>(a.ws.perm), a.ws.xs_hi, a.ws.xs_lo,
                      a.ws.err);
}

cudaError_t launch_expert_gemm(const ExpertArgs& a, int kind, int wfmt, int act, int slot_cap, int num_sms,
                               cudaStream_t s) {
    GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.a = a;
    g.kind = kind;
    g.fmt = wfmt;
    g.act = act;
    g.slot_cap = slot_cap;
    g.planes = (kind == kDown || a.xt == MOE_F32) ? 2 : 1;
    g.nt_max = kBRows / g.planes;
    const int64_t K = (kind == kGateUp) ? a.d : a.f;
    const uint16_t* hi = (kind == kGateUp) ? a.ws.xs_hi : a.ws.h_hi;
    const uint16_t* lo = (kind == kGateUp) ? a.ws.xs_lo : a.ws.h_lo;
    cudaError_t e = plane_map(&g.tb[0], hi, a.P, K);
    if (e == cudaSuccess && g.planes == 2) e = plane_map(&g.tb[1], lo, a.P, K);
    if (e != cudaSuccess) return e;
    const int rows_out = (kind == kGateUp) ? a.rows_gu : a.d;
    const int64_t bound = static_cast<int64_t>(rows_out / kTileM) * (slot_cap + (a.P + g.nt_max - 1) / g.nt_max);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms, bound)));
    return launch_pdl(expert_gemm_kernel, dim3(grid), dim3(kGemmThreads), kGemmSmem, s, g);
}

}  // namespace moe
