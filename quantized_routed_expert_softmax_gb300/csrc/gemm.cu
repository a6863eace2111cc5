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
//   warp 0       weight producer: TMA loads of the raw Q8_0 / NVFP4 bytes of two K steps
//                at a time into a ring of kRawSlots slots.  Tensor maps over the whole expert
//                stack (up to 5-D: byte, row, gate/up half, K panel, expert) make one load
//                of codes and one of scales cover a slot, since every TMA operation has a
//                fixed issue cost of the order of a hundred cycles;
//   warp 1       activation producer: TMA 2-D loads of the token tile's B planes into a
//                ring of kBStages stages of their own, one box per plane whose height is
//                the smallest of kBoxHeights that covers the tile's tokens;
//   warp 2       MMA issuer (one thread): per K step of 64, four K = 16 slices of
//                tcgen05.mma with A read from tensor memory and B from shared memory
//                (A.hi*B.hi, A.lo*B.hi for Q8_0, A.hi*B.lo for two planes; the lo*lo term is
//                below fp32 rounding), committed to the A and B stages' "empty" barriers,
//                and at the end of an item to the accumulator's "full" barrier;
//   warps 4..7   epilogue: tensor memory -> registers (lane quadrant = warp % 4), the
//                activation (SwiGLU pairs gate row i and up row i on accumulator lanes 2i
//                and 2i+1, one shuffle), stores; two accumulators alternate, so the
//                epilogue of one item overlaps the main loop of the next;
//   warps 8..23  dequantisers: raw slot -> f16 A tiles written straight into tensor
//                memory (tcgen05.st; warp w writes lane quadrant w % 4, so it converts
//                rows 32*(w%4).. of one 16-column chunk), which keeps the A operand out of
//                shared memory: shared-memory bandwidth, not the tensor core, bounded the
//                kernel when A went through it.  NVFP4 weights e2m1 * e4m3 are
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

constexpr int kGemmThreads = 768;
constexpr int kTileM = 128;
constexpr int kStepK = 64;                          // one 128-byte swizzle row of f16
constexpr int kBRows = 192;                         // B rows per stage: token tile x planes
constexpr int kSmallTile = 64;                      // tokens per work item, few tokens per expert
constexpr int kLargeTile = 192;                     // ... many tokens per expert (capped by kBRows / planes)
constexpr int kLargeAverage = 96;                   // average tokens per expert that selects large tiles
constexpr int kNumBoxHeights = 3;
constexpr int kBoxHeights[kNumBoxHeights] = {32, 64, 128};   // B box rows (below the tile height)
constexpr int kStepsPerSlot = 2;                    // K steps per raw slot
constexpr int kRawSlots = 4;
constexpr int kMaxAStages = 4;                      // in tensor memory: 64 columns each (hi, lo)
constexpr int kBStages = 6;
constexpr int kRawSlot = 17408;                     // Q8_0: 4 panels x 4096 code bytes + 4 x 256 scale bytes
constexpr int kBStageBytes = kBRows * kStepK * 2;   // 24 KB: B planes
constexpr size_t kGemmSmem = 1024 + static_cast<size_t>(kBStages) * kBStageBytes +
                             static_cast<size_t>(kRawSlots) * kRawSlot;
// Tensor memory: 512 columns of 128 lanes x 32 bits.  A stage s: columns 64*s .. 64*s+31 hold
// the hi part of the K step (two f16 K values per column), 64*s+32 .. the lo part.  Then
// acc_bufs buffers (alternate items) x two issuers' accumulators of acc_stride columns each.
// Two shapes fit: small tiles (4 A stages, 64 tokens, 2 buffers, so the epilogue of one item
// overlaps the next) and large tiles (2 A stages, up to 192 tokens, 1 buffer).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAColsPerStage = 64;

constexpr int kWarpLoadA = 0, kWarpLoadB = 1, kWarpMma = 2, kWarpEpi0 = 4, kWarpConv0 = 8;
constexpr int kConvWarps = 16;

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

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(s_addr(bar)), "r"(n)
                 : "memory");
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
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(s_addr(bar))
                 : "memory");
}

// TMA tile loads of 3, 4 and 5 dimensions (coordinates innermost first), completion on `bar`.
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(s_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                       uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(s_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tma_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                       uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(s_addr(bar))
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

// The same with A in tensor memory (row i in lane i, two K values per 32-bit column).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t v[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
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

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float v[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns of each of the two issuers' accumulators, one wait for both loads.
__device__ __forceinline__ void tmem_ld16x2(uint32_t a0, uint32_t a1, uint32_t r[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
        "[%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(a0), "r"(a1)
        : "memory");
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
    CUtensorMap tb[2][kNumBoxHeights + 1];   // B planes, f16 [P][K] (hi, lo); box 64 columns x bh[i] rows
    CUtensorMap tw_codes, tw_scales;     // the weight stack's codes and scales (see raw_slot_layout)
    ExpertArgs a;
    int kind;            // GemmKind
    int fmt;             // MOE_W_Q8_0 / MOE_W_NVFP4
    int act;             // MOE_ACT_* (gate.up)
    int slot_cap;
    int planes;          // 1 or 2
    int nt_max;          // token tile: kBRows / planes
    int acc_stride;      // tensor-memory columns per accumulator (nt_max rounded up to 32)
    int a_stages;        // A stages in tensor memory (2 or 4)
    int acc_bufs;        // accumulator buffers (1 or 2)
    int nbh;             // box heights in use (kBoxHeights[i] < nt_max, then nt_max itself)
    int bh[kNumBoxHeights + 1];
    uint32_t slot_bytes; // bytes one raw slot receives
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

// raw_slot_layout: what one raw slot (two K steps = 128 columns) holds.
//   Q8_0, K panels of 32 columns: codes [4 panels][128 staged rows][32 B], then scales
//     [4 panels][128][2 B] at byte 16384.
//   NVFP4 K panels of 64 columns: codes [2 panels][128][32 B], then scales [2][128][4 B] at
//     byte 8192.
//   NVFP4 down, neuron layout: codes [8 groups of 16 neurons][16][64 B = the tile's 128 rows,
//     two per byte], then scales [8 groups][128 B] at byte 8192.
// SwiGLU gate.up tiles stage gate rows of 64 neurons as rows 0..63 and the same neurons' up
// rows as 64..127 (the gate/up half is a dimension of the tensor maps).
template <int KIND>
__device__ __forceinline__ void load_slot(const GemmArgs& g, uint32_t dst, int e, int mtile, int ks0, uint64_t* bar) {
    const bool q8 = (g.fmt == MOE_W_Q8_0);
    const uint32_t scales_at = q8 ? 16384u : 8192u;
    if (KIND == kDown && !q8) {
        tma_4d(dst, &g.tw_codes, mtile * 64, 0, ks0 * 4, e, bar);
        tma_3d(dst + scales_at, &g.tw_scales, mtile * kTileM, ks0 * 4, e, bar);
        return;
    }
    const int p0 = ks0 * (q8 ? 2 : 1);   // first K panel
    if (KIND == kGateUp && g.act == MOE_ACT_SWIGLU) {
        tma_5d(dst, &g.tw_codes, 0, mtile * 8, 0, p0, e, bar);
        tma_4d(dst + scales_at, &g.tw_scales, mtile * 64, 0, p0, e, bar);
    } else {
        tma_4d(dst, &g.tw_codes, 0, mtile * (kTileM / 8), p0, e, bar);
        tma_3d(dst + scales_at, &g.tw_scales, mtile * kTileM, p0, e, bar);
    }
}

// Dequantise 16 columns (chunk c16 of K step js of a raw slot) of tile row r into the A hi
// (and, for Q8_0, lo) columns of tensor memory at ta (this warp's lane quadrant).
template <int KIND>
__device__ __forceinline__ void dequant_step(const GemmArgs& g, const unsigned char* raw, int js, uint32_t ta, int r,
                                             int c16) {
    const bool swiglu = (KIND == kGateUp && g.act == MOE_ACT_SWIGLU);
    {
        const int sr = swiglu ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;   // staged row
        uint32_t h[8];
        if (g.fmt == MOE_W_Q8_0) {
            const int pp = 2 * js + (c16 >> 1), hh = c16 & 1;   // panel of 32 columns, half
            const uint4 q = *reinterpret_cast<const uint4*>(raw + pp * 4096 + sr * 32 + hh * 16);
            const unsigned short sbits = *reinterpret_cast<const unsigned short*>(raw + 16384 + pp * 256 + sr * 2);
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
            tmem_st8(ta + 32 + c16 * 8, hl);
        } else if (KIND == kDown) {
            // NVFP4 neuron layout: columns 16*c16 .. +15 are group c16; row sr is nibble
            // (sr & 1) of byte sr/2 in each neuron's run
            const int gg = 4 * js + c16;
            const unsigned char* gb = raw + gg * 1024;
            uint32_t s16;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(static_cast<uint16_t>(raw[8192 + gg * 128 + sr])));
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
            const uint2 cw = *reinterpret_cast<const uint2*>(raw + js * 4096 + sr * 32 + c16 * 8);
            uint32_t s16;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(static_cast<uint16_t>(raw[8192 + js * 512 + sr * 4 + c16])));
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
        tmem_st8(ta + c16 * 8, h);
    }
}

// ------------------------------------------------------------------------------ the kernel
// KIND (gate.up or down) is a template parameter: each launch's code and register allocation
// hold only its own epilogue and conversions.
template <int KIND>
__global__ void __launch_bounds__(kGemmThreads, 1) expert_gemm_kernel(const __grid_constant__ GemmArgs g) {
    pdl_wait();
    const ExpertArgs& a = g.a;
    extern __shared__ __align__(16) unsigned char dsm_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* bstages = base;                                    // kBStages x B planes
    unsigned char* raws = bstages + kBStages * kBStageBytes;          // kRawSlots x kRawSlot
    __shared__ uint64_t raw_full[kRawSlots], raw_empty[kRawSlots];
    __shared__ uint64_t a_full[kMaxAStages], a_empty[kMaxAStages], b_full[kBStages], b_empty[kBStages];
    __shared__ uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t raw_issued[kRawSlots], b_issued[kBStages], a_commits[kMaxAStages], b_commits[kBStages];
    __shared__ uint32_t tmem_base;
    __shared__ int tile_prefix[kMaxE + 1];
    __shared__ int warp_tot[kGemmThreads / 32];
    __shared__ volatile int s_fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t tmem_cols = kTmemCols;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s_addr(&tmem_base)),
                     "r"(tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int s = 0; s < kRawSlots; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], (kConvWarps / 2) * kStepsPerSlot);   // 8 warps per K step
            raw_issued[s] = 0;
        }
        for (int s = 0; s < kMaxAStages; ++s) {
            mbar_init(&a_full[s], kConvWarps / 2);   // one converter group
            mbar_init(&a_empty[s], 1);
            a_commits[s] = 0;
        }
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
            b_issued[s] = 0;
            b_commits[s] = 0;
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 2);   // one commit per issuer
            mbar_init(&acc_empty[s], 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_fail = 0;
    }
    // the work list: per slot, (token tiles) x (row tiles); exclusive prefix over the slots
    const int rows_out = (KIND == kGateUp) ? a.rows_gu : a.d;
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
    const int ksteps = ((KIND == kGateUp) ? a.d : a.f) / kStepK;
    // a_stages (2 or 4) and acc_bufs (1 or 2) are powers of two: shifts and masks
    const uint32_t a_shift = (g.a_stages == 4) ? 2u : 1u, a_mask = (1u << a_shift) - 1u;
    const uint32_t b_shift = (g.acc_bufs == 2) ? 1u : 0u, b_mask = (1u << b_shift) - 1u;
    const uint32_t acc_col0 = static_cast<uint32_t>(g.a_stages) * kAColsPerStage;

    if (warp == kWarpLoadA) {
        // ---------------------------------------------------------------- weight producer
        if (lane == 0) {
            uint32_t sn = 0;   // slots issued
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const Item it = decode_item(g, tile_prefix, mtiles, item);
                for (int ks0 = 0; ks0 < ksteps; ks0 += kStepsPerSlot, ++sn) {
                    const int slot = sn % kRawSlots;
                    const uint32_t use = sn / kRawSlots;
                    if ((use > 0 && !mbar_wait(&raw_empty[slot], use - 1)) || s_fail) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&raw_full[slot], g.slot_bytes);
                    raw_issued[slot] = use + 1;
                    load_slot<KIND>(g, s_addr(raws + slot * kRawSlot), it.e, it.mtile, ks0, &raw_full[slot]);
                }
            }
            if (!ok) {
                s_fail = 1;
                atomicCAS(a.ws.err, 0, kDevErrTimeout);
            }
        }
    } else if (warp == kWarpLoadB) {
        // ---------------------------------------------------------------- activation producer
        if (lane == 0) {
            uint32_t gs = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                const Item it = decode_item(g, tile_prefix, mtiles, item);
                int bi = 0;
                while (bi + 1 < g.nbh && g.bh[bi] < it.nt) ++bi;   // smallest box covering the tile
                const uint32_t bytes = static_cast<uint32_t>(g.bh[bi] * 128 * g.planes);
                for (int ks = 0; ks < ksteps; ++ks, ++gs) {
                    const int st = gs % kBStages;
                    const uint32_t use = gs / kBStages;
                    if ((use > 0 && !mbar_wait(&b_empty[st], use - 1)) || s_fail) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&b_full[st], bytes);
                    b_issued[st] = use + 1;
                    const uint32_t bdst = s_addr(bstages + st * kBStageBytes);
                    for (int p = 0; p < g.planes; ++p)
                        tma_2d(bdst + p * g.nt_max * 128, &g.tb[p][bi], ks * kStepK, it.r_first, &b_full[st]);
                }
            }
            if (!ok) {
                s_fail = 1;
                atomicCAS(a.ws.err, 0, kDevErrTimeout);
            }
        }
    } else if (warp == kWarpMma || warp == kWarpMma + 1) {
        // ---------------------------------------------------------------- MMA issuers
        // Issuer iss takes the K steps whose global index has parity iss (so it always uses A
        // stage iss) and accumulates them into its own accumulator of the item's buffer.
        if (lane == 0) {
            const int iss = warp - kWarpMma;
            const bool alo = (g.fmt == MOE_W_Q8_0);
            const bool two = (g.planes == 2);
            // B descriptors of stage 0; the encoded start address (bits 0..13, bytes / 16) is
            // linear in the address, so stage s adds s * stage bytes / 16 and a K = 16 slice
            // adds 32 bytes (2).  A in tensor memory: a K = 16 slice is 8 columns.
            const uint64_t dB0 = sdesc_k128(s_addr(bstages));
            const uint64_t dBl0 = sdesc_k128(s_addr(bstages + g.nt_max * 128));
            uint32_t gs = 0, n_item = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++n_item) {
                const Item it = decode_item(g, tile_prefix, mtiles, item);
                const uint32_t idesc = idesc_f16((it.nt + 15) & ~15);
                const int buf = static_cast<int>(n_item & b_mask);
                const uint32_t ub = n_item >> b_shift;
                if ((ub > 0 && !mbar_wait(&acc_empty[buf], ub - 1)) || s_fail) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + acc_col0 + static_cast<uint32_t>((2 * buf + iss) * g.acc_stride);
                bool first = true;
                for (int ks = 0; ks < ksteps; ++ks, ++gs) {
                    if ((gs & 1u) != static_cast<uint32_t>(iss)) continue;
                    const int sa = static_cast<int>(gs & a_mask), sb = gs % kBStages;
                    const uint32_t ua = gs >> a_shift, ubb = gs / kBStages;
                    if (!mbar_wait(&a_full[sa], ua) || !mbar_wait(&b_full[sb], ubb) || s_fail) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ta = tmem + static_cast<uint32_t>(sa) * kAColsPerStage;
                    const uint64_t ob = static_cast<uint64_t>(sb * (kBStageBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < kStepK / 16; ++kk) {
                        const uint64_t o = static_cast<uint64_t>(2 * kk);
                        const uint32_t tk = ta + 8 * kk;
                        umma_f16_ta(dt, tk, dB0 + ob + o, idesc, (first && kk == 0) ? 0u : 1u);
                        if (alo) umma_f16_ta(dt, tk + 32, dB0 + ob + o, idesc, 1u);
                        if (two) umma_f16_ta(dt, tk, dBl0 + ob + o, idesc, 1u);
                    }
                    first = false;
                    umma_commit(&a_empty[sa]);
                    umma_commit(&b_empty[sb]);
                    a_commits[sa] = ua + 1;
                    b_commits[sb] = ubb + 1;
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);   // arrives at once when this issuer had no step
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
        const float* ts_arr = (KIND == kGateUp) ? a.gu_ts : a.dn_ts;
        uint32_t n_item = 0, gs0 = 0;   // gs0: global index of the item's first K step
        bool ok = true;
        for (int item = blockIdx.x; item < total; item += gridDim.x, ++n_item, gs0 += ksteps) {
            const Item it = decode_item(g, tile_prefix, mtiles, item);
            const int n16 = (it.nt + 15) & ~15;
            // issuers with at least one K step of this item (both unless it has one step)
            const bool has0 = ksteps >= 2 || (gs0 & 1u) == 0, has1 = ksteps >= 2 || (gs0 & 1u) == 1;
            const int buf = static_cast<int>(n_item & b_mask);
            bool w_ok = mbar_wait(&acc_full[buf], n_item >> b_shift);
            w_ok = __all_sync(0xffffffffu, w_ok) && !s_fail;
            if (!w_ok) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float ts = (g.fmt == MOE_W_NVFP4) ? ts_arr[it.e] : 1.0f;
            const uint32_t tbase =
                tmem + (static_cast<uint32_t>(q * 32) << 16) + acc_col0 + static_cast<uint32_t>(2 * buf * g.acc_stride);
            bool range_ok = true;
            for (int c0 = 0; c0 < n16; c0 += 16) {   // 16 tokens: both accumulators' columns, one wait
                float v[16];
                if (has0 && has1) {
                    uint32_t r[32];
                    tmem_ld16x2(tbase + static_cast<uint32_t>(c0), tbase + static_cast<uint32_t>(g.acc_stride + c0), r);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) v[jj] = __uint_as_float(r[jj]) + __uint_as_float(r[16 + jj]);
                } else {
                    tmem_ld16(tbase + static_cast<uint32_t>(has0 ? c0 : g.acc_stride + c0), v);
                }
                if (KIND == kGateUp && g.act == MOE_ACT_SWIGLU) {
                    // lane pairs (2i: gate row i, 2i+1: up row i) split the 16 tokens: the even
                    // lane takes tokens 0..7 and the odd lane 8..15, each receiving the partner's
                    // half in one shuffle per token; the 8 tokens' steps run side by side
                    const bool odd = lane & 1;
                    float mine[8], u[8];   // this lane's row and the partner's row, of this lane's tokens
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        mine[j] = (odd ? v[8 + j] : v[j]) * ts;
                        u[j] = __shfl_xor_sync(0xffffffffu, (odd ? v[j] : v[8 + j]) * ts, 1);
                    }
                    float hv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) hv[j] = odd ? silu(u[j]) * mine[j] : silu(mine[j]) * u[j];
                    const int64_t col = it.mtile * 64 + (row >> 1);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = c0 + (odd ? 8 : 0) + j;
                        if (n < it.nt) {
                            const int64_t o = static_cast<int64_t>(it.r_first + n) * a.f + col;
                            a.ws.h[o] = hv[j];
                            __half hh, hl;
                            split_f16(hv[j], &hh, &hl);
                            range_ok &= fabsf(hv[j]) <= 65504.0f;
                            a.ws.h_hi[o] = __half_as_ushort(hh);
                            a.ws.h_lo[o] = __half_as_ushort(hl);
                        }
                    }
                } else {
                    // in groups of 8 tokens, each step for all 8 at once, so the tokens' latency
                    // chains overlap
#pragma unroll
                    for (int jb = 0; jb < 16; jb += 8) {
                        float z[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) z[j] = v[jb + j] * ts;
                        if (KIND == kGateUp) {   // ReLU^2
                            const int64_t col = it.mtile * kTileM + row;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int n = c0 + jb + j;
                                const float hv = z[j] > 0.0f ? z[j] * z[j] : 0.0f;
                                if (n < it.nt) {
                                    const int64_t o = static_cast<int64_t>(it.r_first + n) * a.f + col;
                                    a.ws.h[o] = hv;
                                    __half hh, hl;
                                    split_f16(hv, &hh, &hl);
                                    range_ok &= fabsf(hv) <= 65504.0f;
                                    a.ws.h_hi[o] = __half_as_ushort(hh);
                                    a.ws.h_lo[o] = __half_as_ushort(hl);
                                }
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int n = c0 + jb + j;
                                if (n < it.nt)
                                    a.ws.y[static_cast<int64_t>(it.r_first + n) * a.d + it.mtile * kTileM + row] = z[j];
                            }
                        }
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
        // Group grp (8 warps) converts the K steps whose global index has parity grp, so a
        // group's latency (waits, conversion, tensor-memory stores, fences) overlaps the other
        // group's.  Warp w converts lane quadrant w % 4 of two 16-column chunks.
        const int cw = warp - kWarpConv0;
        const int grp = cw / 8;
        const int q = warp & 3;                          // lane quadrant of tensor memory
        const int cpair = (cw % 8) >> 2;                 // chunks 2*cpair, 2*cpair + 1
        const int r = q * 32 + lane;                     // tile row
        const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
        uint32_t gs = 0, sn = 0;   // K steps seen, slots seen
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            for (int ks = 0; ks < ksteps; ++ks, ++gs) {
                const int j = ks % kStepsPerSlot;
                const bool single = (j == 0) && (ks == ksteps - 1);       // a slot holding one K step
                const bool slot_last = (j == kStepsPerSlot - 1) || (ks == ksteps - 1);
                const int slot = sn % kRawSlots;
                const uint32_t slot_use = sn / kRawSlots;
                if (slot_last) ++sn;
                if ((gs & 1u) != static_cast<uint32_t>(grp)) continue;
                const int sa = static_cast<int>(gs & a_mask);
                const uint32_t ua = gs >> a_shift;
                bool w_ok = mbar_wait(&raw_full[slot], slot_use);
                w_ok = w_ok && (ua == 0 || mbar_wait(&a_empty[sa], ua - 1));
                w_ok = __all_sync(0xffffffffu, w_ok) && !s_fail;
                if (!w_ok) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const unsigned char* raw = raws + slot * kRawSlot;
                const uint32_t ta = tq + static_cast<uint32_t>(sa) * kAColsPerStage;
                dequant_step<KIND>(g, raw, j, ta, r, 2 * cpair);
                dequant_step<KIND>(g, raw, j, ta, r, 2 * cpair + 1);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[sa]);
                    mbar_arrive_n(&raw_empty[slot], single ? kStepsPerSlot : 1);
                }
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
        for (int s = 0; s < kBStages; ++s) {
            if (b_issued[s]) ok &= mbar_wait(&b_full[s], b_issued[s] - 1);
            if (b_commits[s]) ok &= mbar_wait(&b_empty[s], b_commits[s] - 1);
        }
        for (int s = 0; s < kMaxAStages; ++s)
            if (a_commits[s]) ok &= mbar_wait(&a_empty[s], a_commits[s] - 1);
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

cudaError_t encode(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUresult r = g_encode(m, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of an f16 plane [rows][cols] (row stride cols*2 bytes), boxes of 64 columns x
// box_rows rows, 128-byte swizzle; rows past the end read as zero.
cudaError_t plane_map(CUtensorMap* m, const uint16_t* base, int64_t rows, int64_t cols, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kStepK), static_cast<cuuint32_t>(box_rows)};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Tensor maps of a stack of E quantised matrices for raw_slot_layout (strides in bytes).
cudaError_t weight_maps(GemmArgs* g, const uint8_t* W, int64_t E, int64_t mat_bytes, int64_t rows_w, int64_t K) {
    const bool q8 = (g->fmt == MOE_W_Q8_0);
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
    const cuuint64_t e64 = static_cast<cuuint64_t>(E), mb = static_cast<cuuint64_t>(mat_bytes);
    if (g->kind == kDown && !q8) {
        // neuron layout: per 16-neuron group, [16 neurons][rows/2 bytes] then [rows] scales
        const int64_t d = rows_w, groups = K / 16, rec = 9 * d;
        const cuuint64_t cd[4] = {static_cast<cuuint64_t>(d / 2), 16, static_cast<cuuint64_t>(groups), e64};
        const cuuint64_t cs[3] = {static_cast<cuuint64_t>(d / 2), static_cast<cuuint64_t>(rec), mb};
        const cuuint32_t cb[4] = {64, 16, 4 * kStepsPerSlot, 1};
        cudaError_t e = encode(&g->tw_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, W, cd, cs, cb, none);
        if (e != cudaSuccess) return e;
        const cuuint64_t sd[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(groups), e64};
        const cuuint64_t ss[2] = {static_cast<cuuint64_t>(rec), mb};
        const cuuint32_t sb[3] = {kTileM, 4 * kStepsPerSlot, 1};
        g->slot_bytes = 64 * 16 * 4 * kStepsPerSlot + kTileM * 4 * kStepsPerSlot;
        return encode(&g->tw_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, W + 8 * d, sd, ss, sb, none);
    }
    // K panels: [rows][32 code bytes] then [rows] scales of 2 (Q8_0) or 4 (NVFP4) bytes.  The
    // codes of 8 consecutive rows are 256 contiguous bytes: that is the innermost box extent,
    // since a copy engine handles a box one innermost run at a time and 32-byte runs left it
    // issuing eight times as many requests for the same bytes.
    const int64_t panel_cols = q8 ? 32 : 64, panels = K / panel_cols;
    const int64_t scb = q8 ? 2 : 4, pbytes = rows_w * (32 + scb);
    const cuuint32_t npan = static_cast<cuuint32_t>((q8 ? 2 : 1) * kStepsPerSlot);
    const CUtensorMapDataType st = q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32;
    g->slot_bytes = npan * (kTileM * 32 + kTileM * static_cast<uint32_t>(scb));
    cudaError_t e;
    if (g->kind == kGateUp && g->act == MOE_ACT_SWIGLU) {
        const int64_t f = rows_w / 2;   // gate rows 0..f-1, up rows f..2f-1
        const cuuint64_t cd[5] = {256, static_cast<cuuint64_t>(f / 8), 2, static_cast<cuuint64_t>(panels), e64};
        const cuuint64_t cs[4] = {256, static_cast<cuuint64_t>(f * 32), static_cast<cuuint64_t>(pbytes), mb};
        const cuuint32_t cb[5] = {256, 8, 2, npan, 1};
        e = encode(&g->tw_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, W, cd, cs, cb, none);
        if (e != cudaSuccess) return e;
        const cuuint64_t sd[4] = {static_cast<cuuint64_t>(f), 2, static_cast<cuuint64_t>(panels), e64};
        const cuuint64_t ss[3] = {static_cast<cuuint64_t>(f * scb), static_cast<cuuint64_t>(pbytes), mb};
        const cuuint32_t sb[4] = {64, 2, npan, 1};
        return encode(&g->tw_scales, st, 4, W + rows_w * 32, sd, ss, sb, none);
    }
    const cuuint64_t cd[4] = {256, static_cast<cuuint64_t>(rows_w / 8), static_cast<cuuint64_t>(panels), e64};
    const cuuint64_t cs[3] = {256, static_cast<cuuint64_t>(pbytes), mb};
    const cuuint32_t cb[4] = {256, kTileM / 8, npan, 1};
    e = encode(&g->tw_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, W, cd, cs, cb, none);
    if (e != cudaSuccess) return e;
    const cuuint64_t sd[3] = {static_cast<cuuint64_t>(rows_w), static_cast<cuuint64_t>(panels), e64};
    const cuuint64_t ss[2] = {static_cast<cuuint64_t>(pbytes), mb};
    const cuuint32_t sb[3] = {kTileM, npan, 1};
    return encode(&g->tw_scales, st, 3, W + rows_w * 32, sd, ss, sb, none);
}

}  // namespace

cudaError_t configure_gemm_kernels() {
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    for (int kind = 0; kind < 2; ++kind) {
        const void* fn = kind == 0 ? reinterpret_cast<const void*>(expert_gemm_kernel<kGateUp>)
                                   : reinterpret_cast<const void*>(expert_gemm_kernel<kDown>);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kGemmSmem));
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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

cudaError_t launch_expert_gemm(const ExpertArgs& a, int kind, int wfmt, int act, int slot_cap, int E, int num_sms,
                               cudaStream_t s) {
    GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.a = a;
    g.kind = kind;
    g.fmt = wfmt;
    g.act = act;
    g.slot_cap = slot_cap;
    g.planes = (kind == kDown || a.xt == MOE_F32) ? 2 : 1;
    // tile shape by the average tokens per active expert
    const bool large = a.P >= static_cast<int64_t>(kLargeAverage) * slot_cap;
    g.nt_max = std::min(large ? kLargeTile : kSmallTile, kBRows / g.planes);
    g.acc_stride = (g.nt_max + 31) & ~31;
    g.acc_bufs = large ? 1 : 2;
    // as many A stages (2 or 4) as tensor memory holds beside the accumulators: with 4, each
    // issuer's next K step can be dequantised while its current one is multiplied
    g.a_stages = (4 * static_cast<int>(kAColsPerStage) + g.acc_bufs * 2 * g.acc_stride <= static_cast<int>(kTmemCols))
                     ? 4 : 2;
    g.nbh = 0;
    for (int i = 0; i < kNumBoxHeights && kBoxHeights[i] < g.nt_max; ++i) g.bh[g.nbh++] = kBoxHeights[i];
    static_assert(kNumBoxHeights + 1 <= 4, "box height table");
    g.bh[g.nbh++] = g.nt_max;
    const int64_t K = (kind == kGateUp) ? a.d : a.f;
    const uint16_t* hi = (kind == kGateUp) ? a.ws.xs_hi : a.ws.h_hi;
    const uint16_t* lo = (kind == kGateUp) ? a.ws.xs_lo : a.ws.h_lo;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < g.nbh && e == cudaSuccess; ++i) {
        e = plane_map(&g.tb[0][i], hi, a.P, K, g.bh[i]);
        if (e == cudaSuccess && g.planes == 2) e = plane_map(&g.tb[1][i], lo, a.P, K, g.bh[i]);
    }
    if (e == cudaSuccess)
        e = (kind == kGateUp) ? weight_maps(&g, a.w_gu, E, a.gu_bytes, a.rows_gu, a.d)
                              : weight_maps(&g, a.w_dn, E, a.dn_bytes, a.d, a.f);
    if (e != cudaSuccess) return e;
    const int rows_out = (kind == kGateUp) ? a.rows_gu : a.d;
    const int64_t bound = static_cast<int64_t>(rows_out / kTileM) * (slot_cap + (a.P + g.nt_max - 1) / g.nt_max);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms, bound)));
    if (kind == kGateUp) return launch_pdl(expert_gemm_kernel<kGateUp>, dim3(grid), dim3(kGemmThreads), kGemmSmem, s, g);
    return launch_pdl(expert_gemm_kernel<kDown>, dim3(grid), dim3(kGemmThreads), kGemmSmem, s, g);
}

}  // namespace moe
