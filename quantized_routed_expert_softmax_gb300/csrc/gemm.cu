// gemm.cu -- expert kernels for many tokens per expert: grouped GEMMs on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// gate.up + activation and the down projection of the routed layer ("Running Gemma 4 26B
// at 5 tokens/s on a 13-year-old Xeon", section "A three-step fix" / "Runtime graph
// fallback": per-expert matmuls over the gate-first/up-second [n_embd, 2*n_ff, n_experts]
// tensor; "Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU", "bytes per token":
// the gateless ReLU^2 latent experts), for batches where each expert sees many tokens.
//
// Swap-AB: D[128 weight rows][N tokens] = W_e[rows][K] * X^T, so the weight rows fill the
// MMA's M = 128 and the expert's tokens (often few) fill N (16..128).  A persistent grid walks
// a device-built list of (expert slot, token tile, row tile) work items.  Per K step of 64:
//   1. raw weight bytes (Q8_0 / NVFP4 panels) and the activation rows stream through a
//      cp.async ring in shared memory (kRaw steps ahead);
//   2. all threads dequantise into f16 tiles in the 128-byte-swizzled K-major layout the
//      tensor core reads and convert the activations to f16.  NVFP4 weights e2m1 * e4m3
//      are exact in f16.  A Q8_0 weight q * d needs up to 18 significant bits, so it is
//      split into hi = f16(q * d) and lo = fma(q, d, -hi) (the exact residual, rounded).
//      bf16 activations in f16's normal range convert exactly; fp32 inputs and the fp32
//      hidden activations are split the same way into hi + lo;
//   3. one thread issues the tcgen05.mma (K = 16 each: A.hi*B.hi, A.lo*B.hi for Q8_0,
//      A.hi*B.lo for fp32 activations; the lo*lo term is below fp32 rounding) into the
//      tensor-memory accumulator and commits them to an mbarrier that frees the stage.
// SwiGLU tiles interleave gate row n and up row n on adjacent accumulator lanes (2i, 2i+1),
// so the epilogue pairs them with one shuffle.  Every wait on an mbarrier is bounded (about
// a second); on timeout the kernel records MOE device error 2, releases its tensor memory
// and returns.
#include "common.cuh"

namespace moe {

constexpr int kGemmThreads = 256;
constexpr int kTileM = 128;
constexpr int kTileN = 128;          // tokens per work item (tensor-memory columns)
constexpr int kStepK = 64;           // one 128-byte swizzle row of f16
constexpr int kRaw = 2;              // raw ring depth (K steps in flight)
constexpr int kStagesMma = 2;        // f16 operand stages
constexpr int kDevErrTimeout = 2;
constexpr long long kWaitLimitNs = 1000000000ll;

// ------------------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t s_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ long long global_ns() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void g_cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void g_cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void g_cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s_addr(bar)), "r"(count) : "memory");
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

// Wait for the phase with the given parity to complete, for at most kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
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

// ------------------------------------------------------------------------------ operands
enum GemmKind { kGateUp = 0, kDown = 1 };

struct GemmArgs {
    ExpertArgs a;
    int kind;          // GemmKind
    int fmt;           // MOE_W_Q8_0 / MOE_W_NVFP4
    int act;           // MOE_ACT_* (gate.up)
    int slot_cap;
};

// Shared-memory plan of one CTA.  Raw slot: A raw bytes (<= 9 KB), then B raw rows
// (<= 128 rows x 256 bytes).  MMA stage: A hi, A lo, B hi, B lo f16 tiles of 16 KB.
constexpr int kRawA = 9216;
constexpr int kRawB = kTileN * kStepK * 4;
constexpr int kRawSlot = kRawA + kRawB;
constexpr int kTileBytes = kTileM * kStepK * 2;     // 16 KB (A, or B with 128 rows)
constexpr int kMmaStage = 4 * kTileBytes;
constexpr size_t kGemmSmem = 1024 + static_cast<size_t>(kRaw) * kRawSlot + static_cast<size_t>(kStagesMma) * kMmaStage;

// The rows of W one work item reads: SwiGLU gate.up tiles take 64 gate rows and the same 64
// neurons' up rows (interleaved in the tile), everything else 128 consecutive rows.
struct RowMap {
    int gate0, up0;    // SwiGLU gate.up
    int row0;          // others
    bool swiglu;
};

// Copy the raw operands of K step `ks` into a raw slot (every thread issues its share).
__device__ __forceinline__ void issue_raw(const GemmArgs& g, unsigned char* raw, const uint8_t* W, int rows_w,
                                          const RowMap& rm, int ks, const int* tok, int nt, int r_first) {
    const ExpertArgs& a = g.a;
    const int tid = threadIdx.x;
    unsigned char* ra = raw;
    unsigned char* rb = raw + kRawA;
    if (g.kind == kDown && g.fmt == MOE_W_NVFP4) {
        // neuron layout: 4 groups of 16 neurons; per group 16 x (64 rows' 32 bytes) then 128 scale bytes
        const int64_t rec = 16 * (a.d / 2) + a.d;
        for (int c = tid; c < 4 * (16 * 4 + 8); c += kGemmThreads) {   // 16-byte chunks
            const int grp = c / 72, rem = c % 72;
            const uint8_t* base = W + (static_cast<int64_t>(ks) * 4 + grp) * rec;
            if (rem < 64) {
                const int n = rem / 4, q = rem % 4;                 // neuron n, rows 32q .. 32q+31 of the tile
                g_cp_async16(s_addr(ra + grp * 1152 + n * 64 + q * 16), base + n * (a.d / 2) + rm.row0 / 2 + q * 16);
            } else {
                const int q = rem - 64;                             // 8 chunks = 128 scale bytes
                g_cp_async16(s_addr(ra + grp * 1152 + 1024 + q * 16), base + 16 * (a.d / 2) + rm.row0 + q * 16);
            }
        }
    } else {
        // K panels: Q8_0 two panels of 32 columns, NVFP4 one panel of 64 columns
        const int npanel = (g.fmt == MOE_W_Q8_0) ? 2 : 1;
        const int64_t pbytes = static_cast<int64_t>(rows_w) * (g.fmt == MOE_W_Q8_0 ? 34 : 36);
        const int scb = (g.fmt == MOE_W_Q8_0) ? 2 : 4;             // scale bytes per row per panel
        const int per_panel = 128 * 32 / 16 + 128 * scb / 16;       // 16-byte chunks
        for (int c = tid; c < npanel * per_panel; c += kGemmThreads) {
            const int p = c / per_panel, rem = c % per_panel;
            const uint8_t* P = W + (static_cast<int64_t>(ks) * npanel + p) * pbytes;
            unsigned char* dst = ra + p * (128 * 32 + 128 * 4);
            if (rem < 256) {       // codes: 128 rows x 32 bytes, 2 chunks per row
                const int r = rem / 2, h = rem % 2;
                const int src_row = rm.swiglu ? ((r < 64) ? rm.gate0 + r : rm.up0 + r - 64) : rm.row0 + r;
                g_cp_async16(s_addr(dst + r * 32 + h * 16), P + static_cast<int64_t>(src_row) * 32 + h * 16);
            } else {               // scales of the same 128 rows (two runs of 64 for SwiGLU)
                const int q = rem - 256;
                const int run_chunks = 64 * scb / 16;
                const int half = q / run_chunks, qi = q % run_chunks;
                const int src_row = rm.swiglu ? (half == 0 ? rm.gate0 : rm.up0) : rm.row0 + 64 * half;
                g_cp_async16(s_addr(dst + 128 * 32 + half * 64 * scb + qi * 16),
                             P + static_cast<int64_t>(rows_w) * 32 + static_cast<int64_t>(src_row) * scb + qi * 16);
            }
        }
    }
    // activations: gate.up reads x rows (bf16: 128 B per step, fp32: 256 B), down reads h rows (fp32)
    const bool f32 = (g.kind == kDown) || a.xt == MOE_F32;
    const int rowbytes = f32 ? 256 : 128;
    const int cpr = rowbytes / 16;
    for (int c = tid; c < nt * cpr; c += kGemmThreads) {
        const int n = c / cpr, q = c % cpr;
        const unsigned char* src;
        if (g.kind == kDown) {
            src = reinterpret_cast<const unsigned char*>(a.ws.h + static_cast<int64_t>(r_first + n) * a.f + ks * kStepK) + q * 16;
        } else if (a.xt == MOE_F32) {
            src = reinterpret_cast<const unsigned char*>(static_cast<const float*>(a.x) + static_cast<int64_t>(tok[n]) * a.d + ks * kStepK) + q * 16;
        } else {
            src = reinterpret_cast<const unsigned char*>(static_cast<const uint16_t*>(a.x) + static_cast<int64_t>(tok[n]) * a.d + ks * kStepK) + q * 16;
        }
        g_cp_async16(s_addr(rb + n * rowbytes + q * 16), src);
    }
}

// Dequantise / convert one K step from a raw slot into an MMA stage.
__device__ __forceinline__ void convert_step(const GemmArgs& g, const unsigned char* raw, unsigned char* st, int nt,
                                             int n16, bool split) {
    const ExpertArgs& a = g.a;
    const int tid = threadIdx.x;
    const unsigned char* ra = raw;
    const unsigned char* rb = raw + kRawA;
    unsigned char* ta = st;
    unsigned char* tal = st + kTileBytes;
    unsigned char* tb = st + 2 * kTileBytes;
    unsigned char* tl = st + 3 * kTileBytes;
    // A: 128 tile rows x 4 chunks of 16 columns
    for (int u = tid; u < kTileM * 4; u += kGemmThreads) {
        const int r = u >> 2, c16 = u & 3;
        // tile row r <- staged row: SwiGLU interleaves gate (staged 0..63) and up (staged 64..127)
        const int sr = (g.kind == kGateUp && g.act == MOE_ACT_SWIGLU) ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;
        uint32_t h[8], hl[8];
        if (g.kind == kDown && g.fmt == MOE_W_NVFP4) {
            // columns 16*c16 .. +15 are group c16 (16 neurons) of this step; row sr
            const unsigned char* gb = ra + c16 * 1152;
            const uint32_t sbyte = gb[1024 + sr];
            uint32_t s16;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(static_cast<uint16_t>(sbyte)));
            const __half sh = __ushort_as_half(static_cast<unsigned short>(s16 & 0xffffu));
            const __half2 s2 = __halves2half2(sh, sh);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // neurons 2j, 2j+1: nibble (sr & 1) of byte sr/2 in each neuron's row run
                const uint32_t b0 = gb[(2 * j) * 64 + (sr >> 1)];
                const uint32_t b1 = gb[(2 * j + 1) * 64 + (sr >> 1)];
                const uint32_t n0 = (sr & 1) ? (b0 >> 4) : (b0 & 0xfu);
                const uint32_t n1 = (sr & 1) ? (b1 >> 4) : (b1 & 0xfu);
                uint32_t h2;
                asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(n0 | (n1 << 4)));
                const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), s2);
                h[j] = *reinterpret_cast<const uint32_t*>(&v);
            }
        } else if (g.fmt == MOE_W_Q8_0) {
            const int p = c16 >> 1, hh = c16 & 1;              // panel of 32 columns, half
            const unsigned char* pan = ra + p * (128 * 32 + 128 * 4);
            const uint4 q = *reinterpret_cast<const uint4*>(pan + sr * 32 + hh * 16);
            const unsigned short sbits = *reinterpret_cast<const unsigned short*>(pan + 128 * 32 + sr * 2);
            const __half2 s2 = __halves2half2(__ushort_as_half(sbits), __ushort_as_half(sbits));
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u8 = w4[i] ^ 0x80808080u;
                const uint32_t lo = __byte_perm(u8, 0x64646464u, 0x4140);
                const uint32_t hi = __byte_perm(u8, 0x64646464u, 0x4342);
                const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
                const __half2 ql = __hsub2(*reinterpret_cast<const __half2*>(&lo), off);   // exact codes
                const __half2 qh = __hsub2(*reinterpret_cast<const __half2*>(&hi), off);
                const __half2 lv = __hmul2(ql, s2), hv = __hmul2(qh, s2);
                const __half2 lr = __hfma2(ql, s2, __hneg2(lv)), hr = __hfma2(qh, s2, __hneg2(hv));
                h[2 * i] = *reinterpret_cast<const uint32_t*>(&lv);
                h[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hv);
                hl[2 * i] = *reinterpret_cast<const uint32_t*>(&lr);
                hl[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hr);
            }
            *reinterpret_cast<uint4*>(tal + swz(r, 2 * c16)) = make_uint4(hl[0], hl[1], hl[2], hl[3]);
            *reinterpret_cast<uint4*>(tal + swz(r, 2 * c16 + 1)) = make_uint4(hl[4], hl[5], hl[6], hl[7]);
        } else {   // NVFP4 K panel of 64 columns: 32 code bytes, 4 scale bytes per row
            const uint2 cw = *reinterpret_cast<const uint2*>(ra + sr * 32 + c16 * 8);
            const uint32_t sbyte = ra[128 * 32 + sr * 4 + c16];
            uint32_t s16;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(static_cast<uint16_t>(sbyte)));
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
    // B: n16 rows (tokens) x 8 chunks of 8 columns; rows >= nt are zero
    const bool f32 = (g.kind == kDown) || a.xt == MOE_F32;
    for (int u = tid; u < n16 * 8; u += kGemmThreads) {
        const int n = u >> 3, c = u & 7;
        uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
        if (n < nt) {
            if (f32) {
                const float4 v0 = *reinterpret_cast<const float4*>(rb + n * 256 + c * 32);
                const float4 v1 = *reinterpret_cast<const float4*>(rb + n * 256 + c * 32 + 16);
                const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const __half2 hh = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
                    const float2 hf = __half22float2(hh);
                    const __half2 ll = __floats2half2_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
                    hw[i] = *reinterpret_cast<const uint32_t*>(&hh);
                    lw[i] = *reinterpret_cast<const uint32_t*>(&ll);
                }
                hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            } else {
                const uint4 b = *reinterpret_cast<const uint4*>(rb + n * 128 + c * 16);
                const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
                uint32_t hw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float f0 = __uint_as_float(bw[i] << 16), f1 = __uint_as_float(bw[i] & 0xffff0000u);
                    const __half2 hh = __floats2half2_rn(f0, f1);
                    hw[i] = *reinterpret_cast<const uint32_t*>(&hh);
                }
                hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
        }
        *reinterpret_cast<uint4*>(tb + swz(n, c)) = hi;
        if (split) *reinterpret_cast<uint4*>(tl + swz(n, c)) = lo;
    }
}

// ------------------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kGemmThreads, 1) expert_gemm_kernel(GemmArgs g) {
    pdl_wait();
    const ExpertArgs& a = g.a;
    extern __shared__ __align__(16) unsigned char dsm_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* rawring = base;
    unsigned char* stages = base + kRaw * kRawSlot;     // kRawSlot is a multiple of 1024
    __shared__ uint64_t bar[kStagesMma];
    __shared__ uint32_t tmem_base;
    __shared__ int tile_prefix[kMaxE + 1];
    __shared__ int tok[kTileN];
    __shared__ int warp_sum[kGemmThreads / 32];
    __shared__ int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // tensor memory: 128 columns (kTileN fp32 accumulators per lane)
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(&tmem_base)),
                     "r"(kTileN));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int s = 0; s < kStagesMma; ++s) mbar_init(&bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_fail = 0;
    }
    // the work list: per slot, (token tiles) x (row tiles); exclusive prefix over the slots
    const int rows_out = (g.kind == kGateUp) ? a.rows_gu : a.d;
    const int mtiles = rows_out / kTileM;
    {
        const int per = (g.slot_cap + kGemmThreads - 1) / kGemmThreads;   // consecutive slots per thread
        const int s0 = tid * per;
        int cnts[4];   // slot_cap <= 1024 = 4 * 256
        int local = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            cnts[i] = 0;
            if (i < per && s0 + i < g.slot_cap) {
                const int c = __ldcg(&a.ws.slot_info[s0 + i].z);
                cnts[i] = ((c + kTileN - 1) / kTileN) * mtiles;
            }
            local += cnts[i];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += warp_sum[w];
        int run = before + incl - local;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
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
    const bool split = (g.kind == kDown) || a.xt == MOE_F32;   // fp32 operands: hi + lo
    const bool alo = (g.fmt == MOE_W_Q8_0);                      // Q8_0 weights: hi + lo
    uint32_t mma_count = 0;   // commits issued by this CTA (stage = count % kStagesMma)

    for (int item = blockIdx.x; item < total && !s_fail; item += gridDim.x) {
        // decode (slot, token tile, row tile)
        int lo = 0, hi = g.slot_cap - 1;
        while (lo < hi) {   // last slot with prefix <= item
            const int mid = (lo + hi + 1) >> 1;
            if (tile_prefix[mid] <= item) lo = mid;
            else hi = mid - 1;
        }
        const int slot = lo;
        const int4 si = __ldcg(a.ws.slot_info + slot);
        const int local = item - tile_prefix[slot];
        const int ntile = local / mtiles, mtile = local % mtiles;
        const int e = si.x, r0 = si.y;
        const int t0 = ntile * kTileN;
        const int nt = min(kTileN, si.z - t0);
        const int n16 = (nt + 15) & ~15;
        const int r_first = r0 + t0;
        RowMap rm;
        rm.swiglu = (g.kind == kGateUp && g.act == MOE_ACT_SWIGLU);
        rm.gate0 = mtile * 64;
        rm.up0 = a.f + mtile * 64;
        rm.row0 = mtile * kTileM;
        const uint8_t* W = (g.kind == kGateUp) ? a.w_gu + static_cast<int64_t>(e) * a.gu_bytes
                                               : a.w_dn + static_cast<int64_t>(e) * a.dn_bytes;
        const int rows_w = (g.kind == kGateUp) ? a.rows_gu : a.d;
        if (g.kind == kGateUp)
            for (int n = tid; n < nt; n += kGemmThreads) tok[n] = slot_token(si, t0 + n, a.ws.perm, a.k);
        __syncthreads();
        // prologue of the raw ring
#pragma unroll
        for (int s = 0; s < kRaw; ++s) {
            if (s < ksteps) issue_raw(g, rawring + s * kRawSlot, W, rows_w, rm, s, tok, nt, r_first);
            g_cp_async_commit();
        }
        const uint32_t idesc = idesc_f16(n16);
        for (int ks = 0; ks < ksteps; ++ks) {
            g_cp_async_wait<kRaw - 1>();
            __syncthreads();
            const uint32_t c = mma_count + ks;
            const int st = c % kStagesMma;
            unsigned char* stg = stages + st * kMmaStage;
            if (c >= kStagesMma) {   // the MMAs that last read this stage are done
                if (!mbar_wait_bounded(&bar[st], ((c / kStagesMma) - 1) & 1)) s_fail = 1;
            }
            convert_step(g, rawring + (ks % kRaw) * kRawSlot, stg, nt, n16, split);
            proxy_fence_smem();
            __syncthreads();
            if (s_fail) break;
            if (ks + kRaw < ksteps)
                issue_raw(g, rawring + (ks % kRaw) * kRawSlot, W, rows_w, rm, ks + kRaw, tok, nt, r_first);
            g_cp_async_commit();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t sa = s_addr(stg), sal = s_addr(stg + kTileBytes);
                const uint32_t sb = s_addr(stg + 2 * kTileBytes), sl = s_addr(stg + 3 * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kStepK / 16; ++kk) {
                    umma_f16(tmem, sdesc_k128(sa + kk * 32), sdesc_k128(sb + kk * 32), idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                    if (alo) umma_f16(tmem, sdesc_k128(sal + kk * 32), sdesc_k128(sb + kk * 32), idesc, 1u);
                    if (split) umma_f16(tmem, sdesc_k128(sa + kk * 32), sdesc_k128(sl + kk * 32), idesc, 1u);
                }
                umma_commit(&bar[st]);
            }
        }
        g_cp_async_wait<0>();
        __syncthreads();
        if (s_fail) break;
        // wait for the item's last commit: every MMA of the item has completed
        {
            const uint32_t c = mma_count + ksteps - 1;
            if (!mbar_wait_bounded(&bar[c % kStagesMma], (c / kStagesMma) & 1)) s_fail = 1;
        }
        mma_count += ksteps;
        tc_fence_after();
        __syncthreads();
        if (s_fail) break;
        // epilogue: warp w reads lanes 32*(w%4).. and columns [(w/4)*64, +64) of the accumulator
        const int q = warp & 3, half = warp >> 2;
        const int row = q * 32 + lane;   // accumulator row = tile row
        for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
            if (c0 >= n16) break;
            float v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), v);
            if (g.kind == kGateUp) {
                const float ts = (g.fmt == MOE_W_NVFP4) ? a.gu_ts[e] : 1.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c0 + j;
                    float z = v[j] * ts;
                    if (g.act == MOE_ACT_SWIGLU) {
                        const float u = __shfl_xor_sync(0xffffffffu, z, 1);   // odd lane holds the up row
                        if (!(lane & 1) && n < nt)
                            a.ws.h[static_cast<int64_t>(r_first + n) * a.f + mtile * 64 + (row >> 1)] = silu(z) * u;
                    } else if (n < nt) {
                        a.ws.h[static_cast<int64_t>(r_first + n) * a.f + mtile * kTileM + row] = z > 0.0f ? z * z : 0.0f;
                    }
                }
            } else {
                const float ts = (g.fmt == MOE_W_NVFP4) ? a.dn_ts[e] : 1.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c0 + j;
                    if (n < nt) a.ws.y[static_cast<int64_t>(r_first + n) * a.d + mtile * kTileM + row] = v[j] * ts;
                }
            }
        }
        tc_fence_before();
        __syncthreads();   // accumulator reads finished before the next item's MMAs
    }
    if (s_fail && tid == 0) atomicCAS(a.ws.err, 0, kDevErrTimeout);
    g_cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTileN));
}

// ------------------------------------------------------------------------------ launchers
cudaError_t configure_gemm_kernels() {
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kGemmSmem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(expert_gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

size_t gemm_smem_bytes() { return kGemmSmem; }

cudaError_t launch_expert_gemm(const ExpertArgs& a, int kind, int wfmt, int act, int slot_cap, int num_sms,
                               cudaStream_t s) {
    GemmArgs g;
    g.a = a;
    g.kind = kind;
    g.fmt = wfmt;
    g.act = act;
    g.slot_cap = slot_cap;
    const int rows_out = (kind == kGateUp) ? a.rows_gu : a.d;
    const int64_t bound = static_cast<int64_t>(rows_out / kTileM) * (slot_cap + (a.P + kTileN - 1) / kTileN);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms, bound)));
    return launch_pdl(expert_gemm_kernel, dim3(grid), dim3(kGemmThreads), kGemmSmem, s, g);
}

}  // namespace moe
