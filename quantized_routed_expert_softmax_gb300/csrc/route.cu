// route.cu -- router projection, top-k + softmax, and the permutation of (token, slot)
// pairs by expert.
//
// Router logits use one canonical fp32 order so that every implementation rounds the
// same way: 256 partial sums (partial l takes i = l, l+256, ... with fused multiply-add,
// increasing i), then a halving tree h = 128..1 (s_l += s_{l+h}).  Thread l of a block
// owns partial l; the tree runs through shared memory down to 32 and then through
// warp shuffles.  Top-k is repeated warp-wide argmax (larger value, then lower index);
// the weights are a softmax over the k selected logits (top-8 of 128 in the Gemma pages,
// top-22 of 512 in the Nemotron page).  The permutation is a stable counting sort of
// the T*k pairs by expert, the grouping an expert-indexed matmul presupposes ("Running
// Gemma 4 26B ... on a 13-year-old Xeon", section "A three-step fix").
#include <algorithm>

#include "common.cuh"

namespace moe {

// ----------------------------------------------------------------------------- logits
// Block: 256 threads (one per partial sum), 4 experts, TT tokens.
template <int TT>
__global__ void __launch_bounds__(256) router_logits_kernel(const void* __restrict__ x, int xt,
                                                             const float* __restrict__ W, int T, int d, int E,
                                                             float* __restrict__ logits) {
    pdl_wait();
    const int l = threadIdx.x;
    const int e0 = blockIdx.x * 4;
    const int t0 = blockIdx.y * TT;
    const int nt = min(TT, T - t0);
    float acc[TT][4];
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

#pragma unroll 4
    for (int i = l; i < d; i += kRouterPartials) {
        const float4 wv = __ldg(reinterpret_cast<const float4*>(W + static_cast<int64_t>(i) * E + e0));
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            if (t < nt) {
                const float xv = load_x(x, xt, static_cast<int64_t>(t0 + t) * d + i);
                acc[t][0] = fmaf(xv, wv.x, acc[t][0]);
                acc[t][1] = fmaf(xv, wv.y, acc[t][1]);
                acc[t][2] = fmaf(xv, wv.z, acc[t][2]);
                acc[t][3] = fmaf(xv, wv.w, acc[t][3]);
            }
        }
    }

    __shared__ float red[TT * 4][kRouterPartials];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c) red[t * 4 + c][l] = acc[t][c];
    __syncthreads();
#pragma unroll
    for (int h = kRouterPartials / 2; h >= 32; h >>= 1) {
        if (l < h) {
#pragma unroll
            for (int v = 0; v < TT * 4; ++v) red[v][l] = red[v][l] + red[v][l + h];
        }
        __syncthreads();
    }
    if (l < 32) {
#pragma unroll
        for (int v = 0; v < TT * 4; ++v) {
            float s = red[v][l];
#pragma unroll
            for (int h = 16; h >= 1; h >>= 1) s = s + __shfl_down_sync(0xffffffffu, s, h);
            const int t = v / 4;
            if (l == 0 && t < nt) logits[static_cast<int64_t>(t0 + t) * E + e0 + (v % 4)] = s;
        }
    }
}

// Many tokens: thread l keeps partial sum l of an 8-token x 8-expert block of logits in
// registers (each x value meets 8 weights and each weight 8 x values).
constexpr int kRtT = 8, kRtE = 8;

__device__ __forceinline__ void rt_cp16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Many tokens, without block barriers in the main loop: warp w owns partial sums
// l = 32w .. 32w+31 and stages its own 32-wide slices of x (8 tokens) and W (8 experts) through a
// private cp.async ring, so a warp waits only for its own copies (__syncwarp).  The W rows of
// a stage are stored with their two 16-byte halves swapped on every other group of 4 rows,
// so that the 128-bit reads of 8 consecutive lanes hit all 32 banks.  The multiply-adds of an
// expert pair go in one packed instruction (x broadcast to both halves, W rows read as pairs):
// each half is the same fmaf step of its own chain.  The block's partials then go through the
// same halving tree as the one-expert kernel above.
template <bool XF32>
__global__ void __launch_bounds__(256, 2) router_logits_warp_kernel(const void* __restrict__ x,
                                                                     const float* __restrict__ W, int T, int d,
                                                                     int E, float* __restrict__ logits) {
    constexpr int kXB = XF32 ? 4 : 2;                     // bytes per x element
    constexpr int kStages = XF32 ? 3 : 4;
    constexpr int kXStage = kRtT * 32 * kXB;              // x slice: [8 tokens][32]
    constexpr int kWStage = 32 * kRtE * 4;                // W slice: [32 rows][8 experts]
    constexpr int kStage = kXStage + kWStage;
    constexpr int kXU = kXStage / 16 / 32;                // 16-byte x copies per lane and stage
    __shared__ __align__(16) unsigned char sm[8 * kStages * kStage];
    static_assert(8 * kStages * kStage >= 32 * kRouterPartials * 4, "tree buffer reuse");
    static_assert(8 * kStages * kStage <= 48 * 1024, "static shared memory");
    pdl_wait();
    const int l = threadIdx.x, warp = l >> 5, lane = l & 31;
    const int e0 = blockIdx.x * kRtE;
    const int t0 = blockIdx.y * kRtT;
    const int nt = min(kRtT, T - t0);
    const int M = d / kRouterPartials;
    unsigned char* ring = sm + warp * kStages * kStage;
    const uint32_t rbase = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    // this lane's copies of a step: their sources advance by 256 columns (x) or rows (W) a step
    const unsigned char* xsrc[kXU];
    uint32_t xdst[kXU];
#pragma unroll
    for (int u = 0; u < kXU; ++u) {
        const int c = lane + 32 * u;
        const int t = c / (kXB * 2), q = c % (kXB * 2);
        const int tt = min(t0 + t, T - 1);
        xsrc[u] = static_cast<const unsigned char*>(x) + (static_cast<int64_t>(tt) * d + warp * 32) * kXB + q * 16;
        xdst[u] = c * 16;
    }
    const float* wsrc[2];
    uint32_t wdst[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {                        // W: 32 rows x 2 halves
        const int c = lane + 32 * u;
        const int r = c >> 1, h = c & 1;
        const int hs = h ^ ((r >> 2) & 1);
        wsrc[u] = W + static_cast<int64_t>(warp * 32 + r) * E + e0 + 4 * h;
        wdst[u] = kXStage + (2 * r + hs) * 16;
    }
    const int64_t wstep = static_cast<int64_t>(kRouterPartials) * E;
    auto issue = [&](int st) {   // the next step's slices into stage st
        const uint32_t dst = rbase + st * kStage;
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            rt_cp16(dst + xdst[u], xsrc[u]);
            xsrc[u] += kRouterPartials * kXB;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            rt_cp16(dst + wdst[u], wsrc[u]);
            wsrc[u] += wstep;
        }
    };
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
        if (st < M) issue(st);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    uint64_t acc[kRtT][kRtE / 2];   // (expert 2p, expert 2p + 1) of token t
#pragma unroll
    for (int t = 0; t < kRtT; ++t)
#pragma unroll
        for (int p = 0; p < kRtE / 2; ++p) acc[t][p] = 0;
    const int sw = (lane >> 2) & 1;
    for (int m0 = 0; m0 < M; m0 += kStages) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) {
            const int m = m0 + st;
            if (m < M) {
                asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
                __syncwarp();
                const unsigned char* xs = ring + st * kStage;
                const ulonglong2* wr = reinterpret_cast<const ulonglong2*>(ring + st * kStage + kXStage) + 2 * lane;
                const ulonglong2 wa = wr[sw], wb = wr[sw ^ 1];
                const uint64_t wp[kRtE / 2] = {wa.x, wa.y, wb.x, wb.y};
#pragma unroll
                for (int t = 0; t < kRtT; ++t) {
                    float xv;
                    if (XF32) xv = reinterpret_cast<const float*>(xs)[t * 32 + lane];
                    else xv = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(xs)[t * 32 + lane]);
                    const uint64_t xx = pack_f32x2(xv, xv);
#pragma unroll
                    for (int p = 0; p < kRtE / 2; ++p) fma_f32x2(acc[t][p], xx, wp[p]);
                }
                __syncwarp();   // every lane is done with the stage before it is refilled
                if (m + kStages < M) issue(st);
                asm volatile("cp.async.commit_group;" ::: "memory");
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // The tree, 32 logits (4 tokens x 8 experts) a pass: thread l stores its 32 partials as 8
    // chunks of 4 logits, chunk u at position u ^ (l & 7) of its 32-float row (16-byte stores
    // and loads without bank conflicts).  Warp w then takes chunk w: lane j loads partials
    // j + 32q (q = 0..7) of its 4 logits, adds levels 128, 64 and 32 in registers (two logits
    // per packed add) and 16 .. 1 with shuffles (lane j adds lane j + h): the same pairs
    // s_l += s_{l+h} in the same order.
    constexpr int kPass = 32;
    float* red = reinterpret_cast<float*>(sm);   // [256 partials][32 logits], chunks swizzled
#pragma unroll
    for (int pass = 0; pass < kRtT * kRtE / kPass; ++pass) {
#pragma unroll
        for (int u = 0; u < kPass / 4; ++u) {   // logits 4u .. 4u+3 of the pass: token t, experts 4(u&1)..
            const int t = pass * (kPass / kRtE) + (u >> 1), p = 2 * (u & 1);
            const float2 a = unpack_f32x2(acc[t][p]), b = unpack_f32x2(acc[t][p + 1]);
            *reinterpret_cast<float4*>(red + l * kPass + 4 * (u ^ (l & 7))) = make_float4(a.x, a.y, b.x, b.y);
        }
        __syncthreads();
        uint64_t sq[8][2];   // partial j + 32q: logits (0, 1) and (2, 3) of the warp's chunk
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int pl = lane + 32 * q;
            const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(red + pl * kPass + 4 * (warp ^ (pl & 7)));
            sq[q][0] = v.x;
            sq[q][1] = v.y;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int q = 0; q < 4; ++q) sq[q][i] = add_f32x2(sq[q][i], sq[q + 4][i]);   // h = 128
            sq[0][i] = add_f32x2(sq[0][i], sq[2][i]);                                    // h = 64
            sq[1][i] = add_f32x2(sq[1][i], sq[3][i]);
            sq[0][i] = add_f32x2(sq[0][i], sq[1][i]);                                    // h = 32
#pragma unroll
            for (int h = 16; h >= 1; h >>= 1) {
                const uint64_t o = __shfl_down_sync(0xffffffffu, sq[0][i], h);
                sq[0][i] = add_f32x2(sq[0][i], o);
            }
        }
        const int t = pass * (kPass / kRtE) + (warp >> 1);
        if (lane == 0 && t < nt) {
            const float2 a = unpack_f32x2(sq[0][0]), b = unpack_f32x2(sq[0][1]);
            float* o = logits + static_cast<int64_t>(t0 + t) * E + e0 + 4 * (warp & 1);
            o[0] = a.x;
            o[1] = a.y;
            o[2] = b.x;
            o[3] = b.y;
        }
        __syncthreads();
    }
}

cudaError_t launch_router_logits(const void* x, int xt, const float* W, int64_t T, int64_t d, int64_t E,
                                 float* logits, cudaStream_t s) {
    const dim3 block(256);
    // (the generic router is also launched with PDL through the helper below)
    const int Ti = (int)T, di = (int)d, Ei = (int)E;
    if (T <= 1) return launch_pdl(router_logits_kernel<1>, dim3(E / 4, 1), block, 0, s, x, xt, W, Ti, di, Ei, logits);
    if (T <= 2) return launch_pdl(router_logits_kernel<2>, dim3(E / 4, 1), block, 0, s, x, xt, W, Ti, di, Ei, logits);
    if (T <= 4) return launch_pdl(router_logits_kernel<4>, dim3(E / 4, 1), block, 0, s, x, xt, W, Ti, di, Ei, logits);
    if (E % 8 == 0) {
        const dim3 grid(static_cast<unsigned>(E / 8), static_cast<unsigned>((T + 7) / 8));
        if (xt == MOE_F32) return launch_pdl(router_logits_warp_kernel<true>, grid, block, 0, s, x, W, Ti, di, Ei, logits);
        return launch_pdl(router_logits_warp_kernel<false>, grid, block, 0, s, x, W, Ti, di, Ei, logits);
    }
    return launch_pdl(router_logits_kernel<8>, dim3(E / 4, (unsigned)((T + 7) / 8)), block, 0, s, x, xt, W, Ti, di, Ei,
                      logits);
}

// ----------------------------------------------------------------------------- top-k
// Warp-wide selection of the best remaining (value, index): larger value, lower index on
// equal values.  Every lane ends with the same winner.
template <int NM>   // E <= 32 * NM
__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ lt, int E, int k, int lane,
                                                  int32_t* my_e, float* my_w) {
    float v[NM];
    uint32_t avail = 0;
#pragma unroll
    for (int m = 0; m < NM; ++m) {
        const int e = lane + 32 * m;
        v[m] = (e < E) ? lt[e] : 0.0f;
        if (e < E) avail |= 1u << m;
    }
    int32_t sel_e = -1;
    float sel_l = 0.0f;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int be = 0x7fffffff;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            if ((avail >> m) & 1u) {
                const int e = lane + 32 * m;
                if (be == 0x7fffffff || v[m] > bv || (v[m] == bv && e < be)) {
                    bv = v[m];
                    be = e;
                }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
        if (lane == j) {
            sel_e = be;
            sel_l = bv;
        }
    }
    const float m0 = __shfl_sync(0xffffffffu, sel_l, 0);
    const float ex = (lane < k) ? expf(sel_l - m0) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    *my_e = sel_e;
    *my_w = (lane < k) ? ex / sum : 0.0f;
}

// Calls f<NM>() with the smallest chunk count NM in {1, 4, 16, 32} that covers E.
template <typename F>
__device__ __forceinline__ void with_chunks(int E, F&& f) {
    if (E <= 32) f(std::integral_constant<int, 1>());
    else if (E <= 128) f(std::integral_constant<int, 4>());
    else if (E <= 512) f(std::integral_constant<int, 16>());
    else f(std::integral_constant<int, 32>());
}

__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                            int32_t* __restrict__ idx, float* __restrict__ w) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    int32_t e;
    float wt;
    with_chunks(E, [&](auto nm) {
        warp_topk_softmax<decltype(nm)::value>(logits + static_cast<int64_t>(t) * E, E, k, lane, &e, &wt);
    });
    if (lane < k) {
        idx[static_cast<int64_t>(t) * k + lane] = e;
        w[static_cast<int64_t>(t) * k + lane] = wt;
    }
}

cudaError_t launch_topk_softmax(const float* logits, int64_t T, int64_t E, int k, int32_t* idx, float* w,
                                cudaStream_t s) {
    const int64_t grid = (T * 32 + 255) / 256;
    return launch_pdl(topk_softmax_kernel, dim3((unsigned)grid), dim3(256), 0, s, logits, (int)T, (int)E, k, idx, w);
}

// ----------------------------------------------------------------------------- permute
// One record per slot once this CTA has written offsets, act_e, perm and n_active (call
// after a __syncthreads): expert, first sorted row, pair count (0 for idle slots), and the
// tokens of its first four rows packed 8 bits each when `pack` (T <= 254).
__device__ void write_slot_infos(int slot_cap, int k, int T, const Workspace& ws, bool pack) {
    const int n_act = *ws.n_active;
    for (int s = threadIdx.x; s < slot_cap; s += blockDim.x) {
        int4 si = make_int4(0, 0, 0, kNoPackedTokens);
        if (s < n_act) {
            const int e = ws.act_e[s];
            const int r0 = ws.offsets[e];
            const int cnt = ws.offsets[e + 1] - r0;
            int packed = kNoPackedTokens;
            if (pack && T <= 254) {
                packed = 0;
                for (int i = 0; i < 4 && i < cnt; ++i) packed |= (ws.perm[r0 + i] / k) << (8 * i);
            }
            si = make_int4(e, r0, cnt, packed);
        }
        ws.slot_info[s] = si;
    }
}

// Exclusive prefix sum over n <= 1024 values held one per thread (blockDim 1024).
__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += n;
        }
        warp_tot[lane] = ti - t;
    }
    __syncthreads();
    const int r = warp_tot[warp] + incl - v;
    __syncthreads();
    return r;
}

// Ranks one chunk of up to 1024 pairs (pairs chunk*1024 .. +1023) in pair order:
// wcnt[w][e] turns into the number of pairs of expert e in warps < w of the chunk, and
// the return value is the pair's rank among its expert's pairs in the chunk.  e = -1
// marks an idle thread.  All threads of the block (1024) must call it.
__device__ __forceinline__ int chunk_rank(int e, int E, int* wcnt /* [32][E] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            const int c = wcnt[w * E + ee];
            wcnt[w * E + ee] = run;
            run += c;
        }
    }
    __syncthreads();
    return e >= 0 ? wcnt[warp * E + e] + rank : 0;
}

// Small problems (T <= 32 tokens, T*k <= 1024 pairs): top-k + softmax (or the supplied
// routing), histogram, scan and stable scatter in one block of 1024 threads.  Also
// builds the list of active experts and clears their group masks.
__global__ void __launch_bounds__(1024) route_small_kernel(const float* __restrict__ logits,
                                                            const int32_t* __restrict__ idx_in,
                                                            const float* __restrict__ w_in, int T, int E, int k,
                                                            int gwords, Workspace ws) {
    pdl_wait();
    extern __shared__ int smem[];
    int* wcnt = smem;                    // [32][E]
    int* sidx = smem + 32 * E;           // [1024]
    int* warp_tot = sidx + 1024;         // [32]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = T * k;

    if (idx_in == nullptr) {
        if (warp < T) {
            int32_t e;
            float wt;
            with_chunks(E, [&](auto nm) {
                warp_topk_softmax<decltype(nm)::value>(logits + static_cast<int64_t>(warp) * E, E, k, lane, &e, &wt);
            });
            if (lane < k) {
                sidx[warp * k + lane] = e;
                ws.idx[warp * k + lane] = e;
                ws.w[warp * k + lane] = wt;
            }
        }
    } else {
        for (int p = threadIdx.x; p < P; p += blockDim.x) {
            int e = idx_in[p];
            if (e < 0 || e >= E) {
                set_error(ws.err, kDevErrBadExpert);
                e = min(max(e, 0), E - 1);
            }
            sidx[p] = e;
            ws.idx[p] = e;
            ws.w[p] = w_in[p];
        }
    }
    __syncthreads();

    const int p = threadIdx.x;
    const int e = (p < P) ? sidx[p] : -1;
    const int local = chunk_rank(e, E, wcnt);
    // per-expert totals (integer shared-memory atomics: the counts do not depend on order)
    __shared__ int tot_sh[kMaxE];
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) tot_sh[ee] = 0;
    __syncthreads();
    if (e >= 0) atomicAdd(&tot_sh[e], 1);
    __syncthreads();
    const int my_tot = (threadIdx.x < E) ? tot_sh[threadIdx.x] : 0;
    const int off = block_exclusive_scan_1024(my_tot, warp_tot);
    const int slot = block_exclusive_scan_1024(my_tot > 0 ? 1 : 0, warp_tot);
    __shared__ int off_sh[kMaxE + 1];
    if (threadIdx.x < E) {
        off_sh[threadIdx.x] = off;
        ws.offsets[threadIdx.x] = off;
        if (my_tot > 0) ws.act_e[slot] = threadIdx.x;
    }
    if (threadIdx.x == E - 1) {
        ws.offsets[E] = off + my_tot;
        *ws.n_active = slot + (my_tot > 0 ? 1 : 0);
    }
    __syncthreads();
    if (e >= 0) {
        const int r = off_sh[e] + local;
        ws.perm[r] = p;
        ws.pos[p] = r;
    }
    const int max_slots = min(E, P);
    for (int i = threadIdx.x; i < max_slots * gwords; i += blockDim.x) ws.gmask[i] = 0;
    __syncthreads();
    write_slot_infos(max_slots, k, T, ws, true);
}

cudaError_t launch_route_small(const float* logits, const int32_t* idx_in, const float* w_in, int64_t T,
                               int64_t E, int k, int gwords, const Workspace& ws, cudaStream_t s) {
    const size_t smem = (32 * (size_t)E + 1024 + 32) * sizeof(int);
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)((32 * kMaxE + 1024 + 32) * sizeof(int)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    return launch_pdl(route_small_kernel, dim3(1), dim3(1024), smem, s, logits, idx_in, w_in, (int)T, (int)E, k, gwords,
                      ws);
}

// Large problems: three kernels over chunks of 1024 pairs.
// (1) rank each pair within its chunk, per-expert chunk counts; copies (clamped) routing.
__global__ void __launch_bounds__(1024) perm_rank_kernel(const int32_t* __restrict__ idx_src,
                                                          const float* __restrict__ w_in, int P, int E,
                                                          Workspace ws) {
    pdl_wait();
    extern __shared__ int wcnt[];   // [32][E]
    const int p = blockIdx.x * 1024 + threadIdx.x;
    int e = -1;
    if (p < P) {
        e = idx_src[p];
        if (e < 0 || e >= E) {
            set_error(ws.err, kDevErrBadExpert);
            e = min(max(e, 0), E - 1);
        }
        if (w_in != nullptr) {           // supplied routing: copy into the workspace
            ws.idx[p] = e;
            ws.w[p] = w_in[p];
        }
    }
    const int local = chunk_rank(e, E, wcnt);
    if (p < P) ws.local_rank[p] = local;
    __syncthreads();
    // chunk totals: count by atomics in shared memory (integer, order-independent)
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x) wcnt[ee] = 0;
    __syncthreads();
    if (e >= 0) atomicAdd(&wcnt[e], 1);
    __syncthreads();
    for (int ee = threadIdx.x; ee < E; ee += blockDim.x)
        ws.chunk_cnt[static_cast<int64_t>(blockIdx.x) * E + ee] = wcnt[ee];
}

// (2) one block: chunk bases, offsets, active list, group-mask clear.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int nchunk, int E, int P, int gwords, Workspace ws) {
    pdl_wait();
    __shared__ int warp_tot[32];
    int total = 0;
    if ((int)threadIdx.x < E) {
        const int ee = threadIdx.x;
        for (int c = 0; c < nchunk; ++c) {
            const int v = ws.chunk_cnt[static_cast<int64_t>(c) * E + ee];
            ws.chunk_cnt[static_cast<int64_t>(c) * E + ee] = total;
            total += v;
        }
    }
    const int off = block_exclusive_scan_1024(total, warp_tot);
    const int slot = block_exclusive_scan_1024(total > 0 ? 1 : 0, warp_tot);
    if ((int)threadIdx.x < E) {
        const int ee = threadIdx.x;
        ws.offsets[ee] = off;
        if (total > 0) ws.act_e[slot] = ee;
        for (int c = 0; c < nchunk; ++c) ws.chunk_cnt[static_cast<int64_t>(c) * E + ee] += off;
        if (ee == E - 1) {
            ws.offsets[E] = off + total;
            *ws.n_active = slot + (total > 0 ? 1 : 0);
        }
    }
    const int max_slots = min(E, P);
    for (int i = threadIdx.x; i < max_slots * gwords; i += blockDim.x) ws.gmask[i] = 0;
    __syncthreads();
    write_slot_infos(max_slots, 0, 0, ws, false);
}

// (3) scatter.
__global__ void __launch_bounds__(256) perm_scatter_kernel(int P, int E, Workspace ws) {
    pdl_wait();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int e = ws.idx[p];
    const int r = ws.chunk_cnt[static_cast<int64_t>(p / 1024) * E + e] + ws.local_rank[p];
    ws.perm[r] = p;
    ws.pos[p] = r;
}

cudaError_t launch_permute_large(const int32_t* idx_in, const float* w_in, int64_t T, int64_t E, int k,
                                 int gwords, const Workspace& ws, cudaStream_t s) {
    const int P = (int)(T * k);
    const int nchunk = (P + 1023) / 1024;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(perm_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(32 * kMaxE * sizeof(int)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int32_t* src = idx_in ? idx_in : ws.idx;
    cudaError_t e = launch_pdl(perm_rank_kernel, dim3(nchunk), dim3(1024), 32 * (size_t)E * sizeof(int), s, src,
                               idx_in ? w_in : nullptr, P, (int)E, ws);
    if (e != cudaSuccess) return e;
    if ((e = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, nchunk, (int)E, P, gwords, ws)) != cudaSuccess)
        return e;
    return launch_pdl(perm_scatter_kernel, dim3((P + 255) / 256), dim3(256), 0, s, P, (int)E, ws);
}

// ----------------------------------------------------------------------------- fused decode routing
// Block-wide exclusive scan (256 threads) over v[0..n), n <= 1024, in place; returns the total.
__device__ __forceinline__ int block_scan_256(int* v, int n, int* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (n + 255) / 256;
    const int b0 = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
        if (b0 + i < n) local += v[b0 + i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            const int c = warp_tot[w];
            warp_tot[w] = run;
            run += c;
        }
        warp_tot[8] = run;
    }
    __syncthreads();
    int run = warp_tot[warp] + incl - local;
    for (int i = 0; i < per; ++i) {
        if (b0 + i < n) {
            const int c = v[b0 + i];
            v[b0 + i] = run;
            run += c;
        }
    }
    const int total = warp_tot[8];
    __syncthreads();
    return total;
}

// Stable permutation of P <= 1024 pairs (expert ids in sidx) by one CTA of 256 threads.
// Writes offsets[E+1], perm, pos, the active-expert list, n_active and the slot records,
// all from values held in shared memory (no read-back of its own global writes).
__device__ void permute_block_256(const int* sidx, int T, int k, int E, int gwords, Workspace ws) {
    const int P = T * k;
    const int slot_cap = min(E, P);
    const bool pack = T <= 254;
    __shared__ int cnt[kMaxE + 1];
    __shared__ int act[kMaxE];
    __shared__ int sperm[1024];
    __shared__ int warp_tot[9];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (P <= 32) {
        // one warp: ranks by direct comparison
        if (warp == 0) {
            const int e = lane < P ? sidx[lane] : 0x7fffffff;
            int before = 0, same_before = 0;
            for (int q = 0; q < P; ++q) {
                const int eq = __shfl_sync(0xffffffffu, e, q);
                before += (eq < e);
                same_before += (eq == e && q < lane);
            }
            const int r = before + same_before;
            if (lane < P) {
                ws.perm[r] = lane;
                ws.pos[lane] = r;
            }
            // lane r takes the expert and the pair at sorted row r
            int se = 0x7fffffff, sp = 0;
            for (int q = 0; q < P; ++q) {
                const int rq = __shfl_sync(0xffffffffu, r, q);
                const int eq = __shfl_sync(0xffffffffu, e, q);
                if (rq == lane) {
                    se = eq;
                    sp = q;
                }
            }
            const int prev = __shfl_up_sync(0xffffffffu, se, 1);
            const bool first = lane < P && (lane == 0 || prev != se);
            const uint32_t fm = __ballot_sync(0xffffffffu, first);
            const int n_act = __popc(fm);
            int packed = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int src = min(lane + i, 31);
                const int tok = __shfl_sync(0xffffffffu, sp, src) / k;
                const int tse = __shfl_sync(0xffffffffu, se, src);
                if (lane + i < P && tse == se) packed |= tok << (8 * i);
            }
            if (first) {
                const int slot = __popc(fm & ((1u << lane) - 1u));
                const uint32_t above = fm & ~((2u << lane) - 1u);
                const int next = above ? (__ffs(above) - 1) : P;
                ws.act_e[slot] = se;
                ws.slot_info[slot] = make_int4(se, lane, next - lane, pack ? packed : kNoPackedTokens);
            }
            for (int sl = n_act + lane; sl < slot_cap; sl += 32) ws.slot_info[sl] = make_int4(0, 0, 0, kNoPackedTokens);
            if (lane == 0) *ws.n_active = n_act;
        }
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            int c = 0;
            for (int q = 0; q < P; ++q) c += (sidx[q] < e);
            ws.offsets[e] = c;
        }
    } else {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) cnt[e] = 0;
        __syncthreads();
        for (int p = threadIdx.x; p < P; p += blockDim.x) atomicAdd(&cnt[sidx[p]], 1);
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) act[e] = cnt[e] > 0 ? 1 : 0;
        __syncthreads();
        block_scan_256(cnt, E, warp_tot);           // cnt -> offsets
        const int n_act = block_scan_256(act, E, warp_tot);
        __shared__ int s_act_e[kMaxE];
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            ws.offsets[e] = cnt[e];
            const int c = ((e + 1 < E) ? cnt[e + 1] : P) - cnt[e];
            if (c > 0) {
                ws.act_e[act[e]] = e;
                s_act_e[act[e]] = e;
            }
        }
        if (threadIdx.x == 0) {
            ws.offsets[E] = P;
            *ws.n_active = n_act;
        }
        __syncthreads();
        // stable ranks: pairs in order, one expert-run counter per expert
        for (int e = threadIdx.x; e < E; e += blockDim.x) act[e] = cnt[e];   // next free row of each expert
        __syncthreads();
        for (int c0 = 0; c0 < P; c0 += 256) {
            const int p = c0 + threadIdx.x;
            const int e = p < P ? sidx[p] : -1;
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            // warps take their turn in order so that rows follow pair order
            for (int w = 0; w < 8; ++w) {
                if (warp == w && e >= 0) {
                    const int r = act[e] + rank;
                    ws.perm[r] = p;
                    ws.pos[p] = r;
                    sperm[r] = p;
                    __syncwarp(peers);
                    if (rank == 0) act[e] += __popc(peers);
                }
                __syncthreads();
            }
        }
        for (int sl = threadIdx.x; sl < slot_cap; sl += blockDim.x) {
            int4 si = make_int4(0, 0, 0, kNoPackedTokens);
            if (sl < n_act) {
                const int e = s_act_e[sl];
                const int r0 = cnt[e];
                const int c = ((e + 1 < E) ? cnt[e + 1] : P) - r0;
                int packed = kNoPackedTokens;
                if (pack) {
                    packed = 0;
                    for (int i = 0; i < 4 && i < c; ++i) packed |= (sperm[r0 + i] / k) << (8 * i);
                }
                si = make_int4(e, r0, c, packed);
            }
            ws.slot_info[sl] = si;
        }
    }
    for (int i = threadIdx.x; i < slot_cap * gwords; i += blockDim.x) ws.gmask[i] = 0;
}

// Router + top-k + softmax + permutation for small batches (T * E <= 4096, T * k <= 1024)
// in one launch.  grid: (32 residue classes, E / (32 * EPL) expert chunks) x 256 threads.
// Warp j of CTA (c, chunk) owns the canonical partial sum l = c + 32 j for the chunk's
// 32 * EPL experts (lane = EPL experts): rows i = l, l + 256, ... of W, staged in shared
// memory with 16-byte asynchronous copies.  Narrow chunks spread the router weights over
// 128-256 CTAs, and the weights come from HBM.  Tree levels h = 128, 64, 32
// combine partials of the same residue c, inside the CTA; the CTA writes its result to
// part[t][e][c].  The last CTA to finish (atomic counter, no waiting) applies levels
// h = 16 .. 1 across the 32 residues, then selects, weights and permutes, and resets the
// counter.
constexpr int kResidues = 32;
constexpr int kFusedRouteLogits = 4096;
constexpr int kRankTopkMaxE = 256;   // above this, top-k goes through segment candidates
constexpr size_t kRouteDecodeMaxSmem = 160 * 1024;   // route_decode_kernel's weight rows and x values (beside 43 KB static)

// a beats b: larger logit, or equal logit and lower expert index
__device__ __forceinline__ bool beats(float va, int ea, float vb, int eb) { return va > vb || (va == vb && ea < eb); }

// Selection, weights and permutation from the logits slog[T][E] in shared memory (every
// thread of the block): top-k with larger first and the lower index on ties, softmax over the
// k selected logits, then the permutation by expert.
// kWarpTopk: the warp-argmax top-k may be chosen (the partial-sum kernel's last CTA; the
// cluster kernel keeps the smaller code of the ranking alone).
template <bool kWarpTopk>
__device__ __forceinline__ void route_select(const float* slog, int T, int E, int k, int gwords, const Workspace& ws) {
    // Top-k: expert e's slot is the number of experts that beat it -- the order repeated
    // selection would produce, computed for all (token, expert) at once.
    __shared__ int sidx[1024];
    __shared__ float stop[1024];
    const int nwarps = static_cast<int>(blockDim.x) >> 5;
    // (measured: a round of the warp argmax costs about a third of one rank item per thread at
    // E = 128, so the warp path is taken when k rounds cost less than the ranking's share)
    const int rank_items = (T * E + static_cast<int>(blockDim.x) - 1) / static_cast<int>(blockDim.x);
    if (kWarpTopk && E <= kRankTopkMaxE && E % 32 == 0 && 2 * T * E > static_cast<int>(blockDim.x) &&
        T <= 4 * nwarps && 2 * 128 * k < 7 * rank_items * E) {
        // one warp per token: k rounds of a warp-wide argmax (larger logit, then lower index),
        // each round's winner taken out -- the order the ranks below give, in k * 5 shuffle steps
        const int lane = threadIdx.x & 31;
        const int per = E / 32;   // logits per lane: experts lane, lane + 32, ...
        for (int t = threadIdx.x >> 5; t < T; t += nwarps) {
            float v[kRankTopkMaxE / 32];
            uint32_t taken = 0;
#pragma unroll
            for (int j = 0; j < kRankTopkMaxE / 32; ++j) v[j] = j < per ? slog[t * E + lane + 32 * j] : 0.0f;
            for (int r = 0; r < k; ++r) {
                float bv = -INFINITY;
                int be = 0x7fffffff;
#pragma unroll
                for (int j = 0; j < kRankTopkMaxE / 32; ++j) {
                    const int e = lane + 32 * j;
                    if (j < per && !((taken >> j) & 1u) && (be == 0x7fffffff || beats(v[j], e, bv, be))) {
                        bv = v[j];
                        be = e;
                    }
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                    if (oe != 0x7fffffff && (be == 0x7fffffff || beats(ov, oe, bv, be))) {
                        bv = ov;
                        be = oe;
                    }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                if (lane == 0) {
                    sidx[t * k + r] = be;
                    stop[t * k + r] = bv;
                }
            }
        }
    } else if (E <= kRankTopkMaxE && 2 * T * E <= static_cast<int>(blockDim.x) && E % 8 == 0) {
        // two threads per (token, expert), each counting over half the experts
        const int it = threadIdx.x >> 1, half = threadIdx.x & 1;
        const bool live = it < T * E;
        const int t = live ? it / E : 0, e = live ? it % E : 0;
        const float v = live ? slog[it] : 0.0f;
        int r[4] = {0, 0, 0, 0};
        if (live) {
            const float4* row = reinterpret_cast<const float4*>(slog + t * E) + half * (E / 8);
            for (int q = 0; q < E / 8; ++q) {
                const float4 o = row[q];
                const int b = 4 * (q + half * (E / 8));
                r[0] += beats(o.x, b, v, e);
                r[1] += beats(o.y, b + 1, v, e);
                r[2] += beats(o.z, b + 2, v, e);
                r[3] += beats(o.w, b + 3, v, e);
            }
        }
        int rank = r[0] + r[1] + r[2] + r[3];
        rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        if (live && half == 0 && rank < k) {
            sidx[t * k + rank] = e;
            stop[t * k + rank] = v;
        }
    } else if (E <= kRankTopkMaxE) {
        for (int it = threadIdx.x; it < T * E; it += blockDim.x) {
            const int t = it / E, e = it % E;
            const float v = slog[it];
            const float4* row = reinterpret_cast<const float4*>(slog + t * E);
            int r[4] = {0, 0, 0, 0};
            for (int q = 0; q < E / 4; ++q) {
                const float4 o = row[q];
                const int b = 4 * q;
                r[0] += beats(o.x, b, v, e);
                r[1] += beats(o.y, b + 1, v, e);
                r[2] += beats(o.z, b + 2, v, e);
                r[3] += beats(o.w, b + 3, v, e);
            }
            const int rank = r[0] + r[1] + r[2] + r[3];
            if (rank < k) {
                sidx[t * k + rank] = e;
                stop[t * k + rank] = v;
            }
        }
    } else {
        // Many experts (then T <= 4096 / E is small): per token, an expert can be among the k
        // best only if fewer than k experts of its own segment (E split into 8) beat it; the
        // experts that beat a top-k member are top-k members themselves, so ranks counted
        // among these candidates are exact for the k best.
        // Each segment's candidates go to fixed slots seg * k + (rank in the segment), so
        // no atomic counter is needed; empty slots hold -1.
        __shared__ int cand_e[8 * kMaxK];
        __shared__ float cand_v[8 * kMaxK];
        const int seg = (E + 7) / 8;
        const int ncs = 8 * k;
        for (int t = 0; t < T; ++t) {
            for (int i = threadIdx.x; i < ncs; i += blockDim.x) cand_e[i] = -1;
            __syncthreads();
            const float* row = slog + t * E;
            for (int e = threadIdx.x; e < E; e += blockDim.x) {
                const float v = row[e];
                const int sg = e / seg, s0 = sg * seg, s1 = min(E, s0 + seg);
                int rank = 0;
#pragma unroll 4
                for (int o = s0; o < s1; ++o) rank += beats(row[o], o, v, e);
                if (rank < k) {
                    cand_e[sg * k + rank] = e;
                    cand_v[sg * k + rank] = v;
                }
            }
            __syncthreads();
            for (int i = threadIdx.x; i < ncs; i += blockDim.x) {
                const int e = cand_e[i];
                if (e < 0) continue;
                const float v = cand_v[i];
                int rank = 0;
#pragma unroll 4
                for (int j = 0; j < ncs; ++j) {
                    const int o = cand_e[j];
                    rank += (o >= 0) && beats(cand_v[j], o, v, e);
                }
                if (rank < k) {
                    sidx[t * k + rank] = e;
                    stop[t * k + rank] = v;
                }
            }
            __syncthreads();
        }
    }
    __syncthreads();
    // softmax over the k selected logits, the maximum (slot 0) subtracted, sum in slot order
    for (int p = threadIdx.x; p < T * k; p += blockDim.x) {
        const int t = p / k;
        const float m0 = stop[t * k];
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) sum += expf(stop[t * k + j] - m0);
        ws.idx[p] = sidx[p];
        ws.w[p] = expf(stop[p] - m0) / sum;
    }
    __syncthreads();
    if (T == 1) {
        // One token, k distinct experts: pair j's sorted row (= its slot) is the number of
        // selected experts with a lower index.
        for (int j = threadIdx.x; j < k; j += blockDim.x) {
            const int e = sidx[j];
            int r = 0;
            for (int i = 0; i < k; ++i) r += sidx[i] < e;
            ws.perm[r] = j;
            ws.pos[j] = r;
            ws.act_e[r] = e;
            ws.slot_info[r] = make_int4(e, r, 1, 0);   // one row: token 0
        }
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            int c = 0;
            for (int i = 0; i < k; ++i) c += sidx[i] < e;
            ws.offsets[e] = c;
        }
        if (threadIdx.x == 0) *ws.n_active = k;
        for (int i = threadIdx.x; i < k * gwords; i += blockDim.x) ws.gmask[i] = 0;
    } else {
        permute_block_256(sidx, T, k, E, gwords, ws);
    }
}

template <int EPL>
__global__ void __launch_bounds__(256) route_decode_kernel(const void* __restrict__ x, int xt,
                                                            const float* __restrict__ W, int T, int d, int E, int k,
                                                            int gwords, Workspace ws) {
    constexpr int kChunk = 32 * EPL;
    const int c = blockIdx.x, chunk = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = chunk * kChunk + lane * EPL;
    const bool on = e0 < E;
    const int nchain = d / kRouterPartials;     // d is a multiple of 256
    // phase 1 uses the buffer as red[8 warps][4 tokens][kChunk experts], the last CTA as the
    // logits slog[T * E]
    __shared__ __align__(16) float buf[kFusedRouteLogits];
    static_assert(8 * 4 * kChunk <= kFusedRouteLogits, "shared buffer reuse");
    float (*red)[4][kChunk] = reinterpret_cast<float (*)[4][kChunk]>(buf);
    float* slog = buf;
    __shared__ int s_last;
    // The CTA's rows of the router weights (warp j: rows l + 256 m, m < nchain, the chunk's
    // experts) are copied into shared memory before waiting for the previous kernel; then the
    // x values the CTA's chains read ([T][8 warps][nchain]).  The products read both from
    // shared memory, so no chain step waits on a global load.
    extern __shared__ __align__(16) float rdyn[];
    float* wsm = rdyn;                                   // [8][nchain][kChunk]
    float* xsm = rdyn + 8 * nchain * kChunk;             // [T][8][nchain]
    {
        const uint32_t wbase = static_cast<uint32_t>(__cvta_generic_to_shared(wsm));
        constexpr int kQ = kChunk / 4;                   // 16-byte pieces of a row segment
        for (int it = threadIdx.x; it < 8 * nchain * kQ; it += blockDim.x) {
            const int ww = it / (nchain * kQ), rem = it % (nchain * kQ);
            const int m = rem / kQ, q4 = rem % kQ;
            const int e = chunk * kChunk + q4 * 4;
            if (e < E) {
                const int64_t i = c + 32 * ww + static_cast<int64_t>(kRouterPartials) * m;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(wbase + static_cast<uint32_t>(it) * 16),
                             "l"(W + i * E + e)
                             : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    pdl_wait();
    // No early trigger: the expert kernel that follows is launched once the partial-sum CTAs
    // have exited (and the last one triggers below), so its CTAs spread over every SM
    // instead of piling onto the few SMs the routing CTAs leave free.
    for (int it = threadIdx.x; it < T * 8 * nchain; it += blockDim.x) {
        const int t = it / (8 * nchain), rem = it % (8 * nchain);
        const int ww = rem / nchain, m = rem % nchain;
        xsm[it] = load_x(x, xt, static_cast<int64_t>(t) * d + c + 32 * ww + static_cast<int64_t>(kRouterPartials) * m);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const float* wrow = wsm + warp * nchain * kChunk + lane * EPL;
    for (int t0 = 0; t0 < T; t0 += 4) {
        const int nt = min(4, T - t0);
        float acc[4][EPL];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int q = 0; q < EPL; ++q) acc[t][q] = 0.0f;
        if (on) {
            const float* xr = xsm + (t0 * 8 + warp) * nchain;
            for (int m = 0; m < nchain; ++m) {   // chain l: fmaf over i = l, l + 256, ... in increasing i
                float wv[EPL];
#pragma unroll
                for (int q = 0; q < EPL; ++q) wv[q] = wrow[m * kChunk + q];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float xv = (t < nt) ? xr[t * 8 * nchain + m] : 0.0f;
#pragma unroll
                    for (int q = 0; q < EPL; ++q) acc[t][q] = fmaf(xv, wv[q], acc[t][q]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int q = 0; q < EPL; ++q) red[warp][t][lane * EPL + q] = acc[t][q];
        __syncthreads();
        // levels h = 128, 64, 32: warp j += warp j + h/32 (same residue c)
        for (int it = threadIdx.x; it < 4 * kChunk; it += blockDim.x) {
            const int t = it / kChunk, ee = it % kChunk;
            float sv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) sv[j] = red[j][t][ee];
#pragma unroll
            for (int j = 0; j < 4; ++j) sv[j] = sv[j] + sv[j + 4];
#pragma unroll
            for (int j = 0; j < 2; ++j) sv[j] = sv[j] + sv[j + 2];
            sv[0] = sv[0] + sv[1];
            const int e = chunk * kChunk + ee;
            if (t < nt && e < E) ws.rpart[(static_cast<int64_t>(t0 + t) * E + e) * kResidues + c] = sv[0];
        }
        __syncthreads();
    }
    // the last CTA to finish does the rest
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = (atomicAdd(ws.route_ctr, 1) == static_cast<int>(gridDim.x * gridDim.y) - 1);
    __syncthreads();
    if (!s_last) return;
    pdl_trigger();   // the expert kernel's launch overlaps this CTA's selection and permutation
    __threadfence();
    // levels h = 16 .. 1 across the 32 residues; two logits per thread with all their loads
    // issued before either tree
    for (int it0 = threadIdx.x; it0 < T * E; it0 += 2 * blockDim.x) {
        float sv[2][kResidues];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int it = it0 + u * blockDim.x;
            if (it < T * E) {
                const float4* pp = reinterpret_cast<const float4*>(ws.rpart + static_cast<int64_t>(it) * kResidues);
#pragma unroll
                for (int q = 0; q < kResidues / 4; ++q) {
                    const float4 v = __ldcg(pp + q);
                    sv[u][4 * q] = v.x, sv[u][4 * q + 1] = v.y, sv[u][4 * q + 2] = v.z, sv[u][4 * q + 3] = v.w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int it = it0 + u * blockDim.x;
            if (it < T * E) {
#pragma unroll
                for (int h = kResidues / 2; h >= 1; h >>= 1)
#pragma unroll
                    for (int j = 0; j < h; ++j) sv[u][j] = sv[u][j] + sv[u][j + h];
                slog[it] = sv[u][0];
                ws.logits[it] = sv[u][0];
            }
        }
    }
    __syncthreads();
    route_select<true>(slog, T, E, k, gwords, ws);
    if (threadIdx.x == 0) *ws.route_ctr = 0;
}

// The same computation for one to a few tokens as ONE thread-block cluster of E / EPC CTAs
// (at most 16): CTA g owns experts [g * EPC, (g + 1) * EPC) and thread l the canonical
// partial sum l (i = l, l + 256, ...).  The CTA's slice of the router weights does not
// depend on the previous kernel, so it is copied into shared memory before waiting for it.
// After the fixed halving tree (h = 128, 64, 32 through shared memory, 16 .. 1 by warp
// shuffles) the CTA writes its logits straight into the shared memory of CTA 0 of the
// cluster (distributed shared memory); one cluster barrier later CTA 0 has every logit and
// selects, weights and permutes.  Compared with per-CTA partials in global memory and a
// "last CTA" counter, this takes a global round trip, an atomic and a grid-wide fence off the
// serial path of every decode step.
constexpr int kClusterMaxAcc = 32;   // T * EPC accumulators per thread
constexpr int kClusterMaxCtas = 16;
constexpr size_t kClusterMaxDynSmem = 200 * 1024;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared-memory address of the same variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// 16-byte chunk q of weight row i sits at chunk q ^ wsw<EPC>(i): the rows that the 8 lanes
// of one shared-memory wavefront read then fall on distinct banks.
template <int EPC>
__device__ __forceinline__ int wsw(int i) {
    constexpr int cpr = EPC / 4;
    return (i / (8 / cpr)) & (cpr - 1);
}

template <int EPC>
__global__ void __launch_bounds__(256, 1) route_cluster_kernel(const void* __restrict__ x, int xt,
                                                               const float* __restrict__ W, int T, int d, int E,
                                                               int k, int gwords, Workspace ws) {
    constexpr int TT = kClusterMaxAcc / EPC;   // tokens at most
    constexpr int cpr = EPC / 4;                // 16-byte chunks per weight row
    extern __shared__ __align__(16) float csm[];
    float* wsl = csm;                                             // [d][EPC], chunk-swizzled
    float* red = csm;                                             // after the products: tree
    float* slog = csm + ((d * EPC > 192 * kClusterMaxAcc) ? d * EPC : 192 * kClusterMaxAcc);   // [T][E]
    float* xs = slog + T * E;                                     // [T][d]
    const uint32_t g = cluster_ctarank();
    const int l = threadIdx.x;
    cluster_arrive_relaxed();   // every CTA of the cluster has started before any remote store
    {
        const uint32_t wb = static_cast<uint32_t>(__cvta_generic_to_shared(wsl));
        const float* src = W + static_cast<int64_t>(g) * EPC;
        for (int c = l; c < d * cpr; c += 256) {
            const int i = c / cpr, q = c % cpr;
            rt_cp16(wb + static_cast<uint32_t>((i * cpr + (q ^ wsw<EPC>(i))) * 16), src + static_cast<int64_t>(i) * E + 4 * q);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    pdl_wait();
    // x rows into shared memory as fp32: one round trip for all of them
    if (xt == MOE_F32) {
        const float4* src = static_cast<const float4*>(x);
        for (int i = l; i < T * d / 4; i += 256) reinterpret_cast<float4*>(xs)[i] = __ldg(src + i);
    } else {
        const uint4* src = static_cast<const uint4*>(x);   // 8 bf16
        for (int i = l; i < T * d / 8; i += 256) {
            const uint4 v = __ldg(src + i);
            float4* o = reinterpret_cast<float4*>(xs) + 2 * i;
            o[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                               __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
            o[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                               __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int nchain = d / kRouterPartials;
    float acc[TT][EPC];
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[t][e] = 0.0f;
#pragma unroll 4
    for (int m = 0; m < nchain; ++m) {
        const int i = l + m * kRouterPartials;
        const float4* row = reinterpret_cast<const float4*>(wsl) + i * cpr;
        float wv[EPC];
#pragma unroll
        for (int q = 0; q < cpr; ++q) {
            const float4 v = row[q ^ wsw<EPC>(i)];
            wv[4 * q] = v.x, wv[4 * q + 1] = v.y, wv[4 * q + 2] = v.z, wv[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int t = 0; t < TT; ++t)
            if (t < T) {
                const float xv = xs[t * d + i];
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[t][e] = fmaf(xv, wv[e], acc[t][e]);
            }
    }
    // levels h = 128, 64, 32: s_l += s_{l+h} through shared memory (the weight slice is dead);
    // red[j][0..h) for accumulator j, two regions so that one barrier separates the levels
    __syncthreads();
    {
        float* r0 = red;                              // [32][128]
        float* r1 = red + 128 * kClusterMaxAcc;       // [32][64]
#pragma unroll
        for (int lev = 0; lev < 3; ++lev) {
            const int h = 128 >> lev;
            float* rb = (lev == 1) ? r1 : r0;
            if (l >= h && l < 2 * h) {
#pragma unroll
                for (int t = 0; t < TT; ++t)
                    if (t < T)
#pragma unroll
                        for (int e = 0; e < EPC; ++e) rb[(t * EPC + e) * h + (l - h)] = acc[t][e];
            }
            __syncthreads();
            if (l < h) {
#pragma unroll
                for (int t = 0; t < TT; ++t)
                    if (t < T)
#pragma unroll
                        for (int e = 0; e < EPC; ++e) acc[t][e] = acc[t][e] + rb[(t * EPC + e) * h + l];
            }
        }
    }
    cluster_wait_acquire();   // (the barrier armed at entry): CTA 0's shared memory is live
    if (l < 32) {
        // levels h = 16 .. 1 across the lanes; lane 0 ends with s_0 of every accumulator
#pragma unroll
        for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < T)
#pragma unroll
                    for (int e = 0; e < EPC; ++e)
                        acc[t][e] = acc[t][e] + __shfl_down_sync(0xffffffffu, acc[t][e], h);
        if (l == 0) {
            const uint32_t dst = cluster_map(slog, 0);
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < T)
#pragma unroll
                    for (int e = 0; e < EPC; ++e)
                        cluster_st_f32(dst + static_cast<uint32_t>((t * E + static_cast<int>(g) * EPC + e) * 4), acc[t][e]);
        }
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    if (g != 0) return;
    pdl_trigger();   // the expert kernel's launch overlaps the selection and permutation
    for (int it = l; it < T * E; it += blockDim.x) ws.logits[it] = slog[it];
    route_select<false>(slog, T, E, k, gwords, ws);
}

// Experts per CTA of the cluster kernel for E experts (0: not eligible).
int route_cluster_epc(int64_t E) {
    for (int epc : {4, 8, 16, 32})
        if (E % epc == 0 && E / epc <= kClusterMaxCtas) return epc;
    return 0;
}

size_t route_cluster_smem(int64_t T, int64_t d, int64_t E, int epc) {
    const int64_t tree = 192 * kClusterMaxAcc;
    return static_cast<size_t>(std::max<int64_t>(d * epc, tree) + T * E + T * d) * sizeof(float);
}

bool g_route_cluster_ok = false;

template <int EPC>
cudaError_t configure_route_cluster() {
    cudaError_t e = cudaFuncSetAttribute(route_cluster_kernel<EPC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(route_cluster_kernel<EPC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kClusterMaxDynSmem));
    return e;
}

// Enables the cluster router when a 16-CTA cluster with the largest shared-memory request
// can be resident; otherwise every shape keeps the partial-sum router.
cudaError_t configure_route_kernels() {
    // route_decode_kernel: its weight rows and x values, up to kRouteDecodeMaxSmem (larger
    // shapes take the many-token routing kernels)
    for (const void* fn : {reinterpret_cast<const void*>(route_decode_kernel<1>),
                           reinterpret_cast<const void*>(route_decode_kernel<2>),
                           reinterpret_cast<const void*>(route_decode_kernel<4>)}) {
        const cudaError_t ea = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    static_cast<int>(kRouteDecodeMaxSmem));
        if (ea != cudaSuccess) return ea;
    }
    cudaError_t e = configure_route_cluster<4>();
    if (e == cudaSuccess) e = configure_route_cluster<8>();
    if (e == cudaSuccess) e = configure_route_cluster<16>();
    if (e == cudaSuccess) e = configure_route_cluster<32>();
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        g_route_cluster_ok = false;
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterMaxCtas);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = kClusterMaxDynSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterMaxCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, route_cluster_kernel<8>, &cfg);
    g_route_cluster_ok = (e == cudaSuccess && n >= 1);
    (void)cudaGetLastError();
    return cudaSuccess;
}

template <int EPC>
cudaError_t launch_route_cluster(const void* x, int xt, const float* W, int T, int d, int E, int k, int gwords,
                                 const Workspace& ws, size_t smem, cudaStream_t s) {
    const unsigned ctas = static_cast<unsigned>(E / EPC);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, route_cluster_kernel<EPC>, x, xt, W, T, d, E, k, gwords, ws);
}

// Dynamic shared memory of route_decode_kernel: the CTA's router-weight rows and x values.
size_t route_decode_smem(int64_t T, int64_t d, int epl) {
    const int64_t nchain = d / kRouterPartials;
    return static_cast<size_t>(8 * nchain * 32 * epl + T * 8 * nchain) * sizeof(float);
}

int route_decode_epl(int64_t E) { return (E <= 128) ? 1 : (E <= 512 ? 2 : 4); }

// Whether the one-launch routing serves T tokens of this shape (the cluster kernel, or the
// partial-sum kernel whose shared memory holds its weight rows and x values).
bool route_decode_fits(int64_t T, int64_t d, int64_t E) {
    const int epc = route_cluster_epc(E);
    if (epc > 0 && T * epc <= kClusterMaxAcc && route_cluster_smem(T, d, E, epc) <= kClusterMaxDynSmem) return true;
    return route_decode_smem(T, d, route_decode_epl(E)) <= kRouteDecodeMaxSmem;
}

cudaError_t launch_route_decode(const void* x, int xt, const float* W, int64_t T, int64_t d, int64_t E, int k,
                                int gwords, const Workspace& ws, cudaStream_t s) {
    const int epc = route_cluster_epc(E);
    if (g_route_cluster_ok && epc > 0 && T * epc <= kClusterMaxAcc) {
        const size_t smem = route_cluster_smem(T, d, E, epc);
        if (smem <= kClusterMaxDynSmem) {
            const int Tc = static_cast<int>(T), dc = static_cast<int>(d), Ec = static_cast<int>(E);
            switch (epc) {
                case 4: return launch_route_cluster<4>(x, xt, W, Tc, dc, Ec, k, gwords, ws, smem, s);
                case 8: return launch_route_cluster<8>(x, xt, W, Tc, dc, Ec, k, gwords, ws, smem, s);
                case 16: return launch_route_cluster<16>(x, xt, W, Tc, dc, Ec, k, gwords, ws, smem, s);
                default: return launch_route_cluster<32>(x, xt, W, Tc, dc, Ec, k, gwords, ws, smem, s);
            }
        }
    }
    // experts per lane: chunks narrow enough that the router weights spread over >= 128 CTAs
    const int epl = route_decode_epl(E);
    const dim3 grid(kResidues, static_cast<unsigned>((E + 32 * epl - 1) / (32 * epl)));
    const int Ti = static_cast<int>(T), di = static_cast<int>(d), Ei = static_cast<int>(E);
    const size_t smem = route_decode_smem(T, d, epl);
    if (epl == 1) return launch_pdl(route_decode_kernel<1>, grid, dim3(256), smem, s, x, xt, W, Ti, di, Ei, k, gwords, ws);
    if (epl == 2) return launch_pdl(route_decode_kernel<2>, grid, dim3(256), smem, s, x, xt, W, Ti, di, Ei, k, gwords, ws);
    return launch_pdl(route_decode_kernel<4>, grid, dim3(256), smem, s, x, xt, W, Ti, di, Ei, k, gwords, ws);
}

}  // namespace moe
