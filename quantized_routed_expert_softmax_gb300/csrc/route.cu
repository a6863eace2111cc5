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
#include "common.cuh"

namespace moe {

// ----------------------------------------------------------------------------- logits
// Block: 256 threads (one per partial sum), 4 experts, TT tokens.
template <int TT>
__global__ void __launch_bounds__(256) router_logits_kernel(const void* __restrict__ x, int xt,
                                                             const float* __restrict__ W, int T, int d, int E,
                                                             float* __restrict__ logits) {
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

cudaError_t launch_router_logits(const void* x, int xt, const float* W, int64_t T, int64_t d, int64_t E,
                                 float* logits, cudaStream_t s) {
    const dim3 block(256);
    if (T <= 1) {
        router_logits_kernel<1><<<dim3(E / 4, T), block, 0, s>>>(x, xt, W, (int)T, (int)d, (int)E, logits);
    } else if (T <= 2) {
        router_logits_kernel<2><<<dim3(E / 4, 1), block, 0, s>>>(x, xt, W, (int)T, (int)d, (int)E, logits);
    } else if (T <= 4) {
        router_logits_kernel<4><<<dim3(E / 4, 1), block, 0, s>>>(x, xt, W, (int)T, (int)d, (int)E, logits);
    } else {
        router_logits_kernel<8><<<dim3(E / 4, (unsigned)((T + 7) / 8)), block, 0, s>>>(x, xt, W, (int)T, (int)d,
                                                                                        (int)E, logits);
    }
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- top-k
// Warp-wide selection of the best remaining (value, index): larger value, lower index on
// equal values.  Every lane ends with the same winner.
__device__ __forceinline__ void warp_topk_softmax(const float* __restrict__ lt, int E, int k, int lane,
                                                  int32_t* my_e, float* my_w) {
    float v[kMaxE / 32];
    uint32_t avail = 0;
#pragma unroll
    for (int m = 0; m < kMaxE / 32; ++m) {
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
        for (int m = 0; m < kMaxE / 32; ++m) {
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

__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                            int32_t* __restrict__ idx, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    int32_t e;
    float wt;
    warp_topk_softmax(logits + static_cast<int64_t>(t) * E, E, k, lane, &e, &wt);
    if (lane < k) {
        idx[static_cast<int64_t>(t) * k + lane] = e;
        w[static_cast<int64_t>(t) * k + lane] = wt;
    }
}

cudaError_t launch_topk_softmax(const float* logits, int64_t T, int64_t E, int k, int32_t* idx, float* w,
                                cudaStream_t s) {
    const int64_t grid = (T * 32 + 255) / 256;
    topk_softmax_kernel<<<(unsigned)grid, 256, 0, s>>>(logits, (int)T, (int)E, k, idx, w);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- permute
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
            warp_topk_softmax(logits + static_cast<int64_t>(warp) * E, E, k, lane, &e, &wt);
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
    route_small_kernel<<<1, 1024, smem, s>>>(logits, idx_in, w_in, (int)T, (int)E, k, gwords, ws);
    return cudaGetLastError();
}

// Large problems: three kernels over chunks of 1024 pairs.
// (1) rank each pair within its chunk, per-expert chunk counts; copies (clamped) routing.
__global__ void __launch_bounds__(1024) perm_rank_kernel(const int32_t* __restrict__ idx_src,
                                                          const float* __restrict__ w_in, int P, int E,
                                                          Workspace ws) {
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
}

// (3) scatter.
__global__ void __launch_bounds__(256) perm_scatter_kernel(int P, int E, Workspace ws) {
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
    perm_rank_kernel<<<nchunk, 1024, 32 * (size_t)E * sizeof(int), s>>>(src, idx_in ? w_in : nullptr, P, (int)E,
                                                                        ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    perm_scan_kernel<<<1, 1024, 0, s>>>(nchunk, (int)E, P, gwords, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    perm_scatter_kernel<<<(P + 255) / 256, 256, 0, s>>>(P, (int)E, ws);
    return cudaGetLastError();
}

}  // namespace moe
