// gemv.cu -- expert kernels for a few tokens per expert: weight-streaming GEMVs.
//
// gate.up (+ activation): "Running Gemma 4 26B at 5 tokens/s on a 13-year-old Xeon",
//   section "A three-step fix" / "Runtime graph fallback": the fused [n_embd, 2*n_ff,
//   n_experts] tensor, gate rows first and up rows second, then SiLU(gate)*up; or the
//   gateless latent expert with ReLU^2 ("Running NVIDIA's new 120B Nemotron-3.5-Super
//   on an 8GB GPU", "bytes per token").
// down: the same Nemotron page, "How the engine works", step 4: only 16-neuron groups
//   holding a non-zero activation are read.
// combine: same page, "How we check correctness": per-(token, expert) results summed in
//   a fixed order instead of scatter-add atomics.
//
// Layout in HBM (include/moe.h): weights in K panels, so that lane l of a warp owns one
// weight row and streams it 32 bytes per panel; a warp reads 1 KB contiguous per panel
// and no cross-lane reduction is needed.  The 8 warps of a CTA split the K panels of its
// rows; each warp issues the loads of all its panels (up to a batch of 12) before it
// waits on any of them, so a CTA keeps its whole weight slice in flight.  Partial sums
// meet in shared memory in a fixed warp order: results are bitwise reproducible.
// Dequantisation is exact (int8 or e2m1 codes times the block scale); accumulation is
// fp32; the tokens of one expert sit in shared memory as fp32.
#include "gemv_core.cuh"

namespace moe {


// Stream panels [pb, pe) (restricted to `active` ones when gm != nullptr) through the
// warp's ring and accumulate.
template <int FMT, typename Between>
__device__ __forceinline__ void stream_panels(const uint8_t* W, int rows, int rowA, int rowB, int pb, int pe,
                                              unsigned char* ring, const __half* xs, int ld, int nt,
                                              const uint32_t* gm, float acc[2][4], bool split, int lo_off,
                                              Between&& between) {
    const uint64_t pol = l2_evict_first_policy();
    auto skip_of = [&](int b) -> int {
        if (!gm) return 0;
        const int g = 2 * b;
        return (((gm[g >> 5] >> (g & 31)) & 1u) ? 0 : 1) | (((gm[(g + 1) >> 5] >> ((g + 1) & 31)) & 1u) ? 0 : 2);
    };
    auto next = [&](int b) {
        while (b < pe && skip_of(b) == 3) ++b;
        return b;
    };
    int bi = next(pb);
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
        if (bi < pe) {
            issue_panel_block<FMT>(smem_addr(ring + s * kSlotBytes), W, rows, rowA, rowB, bi, pol, skip_of(bi));
            bi = next(bi + 1);
        }
        cp_async_commit();
    }
    between();   // block-wide: stage the activations while the first copies are in flight
    int bc = next(pb);
    for (int i = 0; bc < pe; ++i) {
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const int s = i % kStages;
        panel_mma<FMT>(ring + s * kSlotBytes, xs, ld, bc, nt, skip_of(bc), acc, split, lo_off);
        __syncwarp();   // every lane is done with the slot before it is refilled
        if (bi < pe) {
            issue_panel_block<FMT>(smem_addr(ring + s * kSlotBytes), W, rows, rowA, rowB, bi, pol, skip_of(bi));
            bi = next(bi + 1);
        }
        cp_async_commit();
        bc = next(bc + 1);
    }
}

// The same stream for the dense gate.up panels (no group skips), with the bookkeeping cut
// to the bone: per-lane source pointers advanced by one add per panel, and the ring unrolled
// so that every slot offset is a constant.  The per-panel arithmetic (conversion, MMAs, scale
// FMAs) is a third of the instructions the general loop spends per panel; the rest was
// address and loop overhead, and the SMs were issue-bound.
template <int FMT, typename Between>
__device__ __forceinline__ void stream_panels_dense(const uint8_t* W, int rows, int rowA, int rowB, int pb, int pe,
                                                    unsigned char* ring, const __half* xs, int ld, int nt,
                                                    float acc[2][4], bool split, int lo_off, Between&& between) {
    const int lane = threadIdx.x & 31;
    const uint64_t pol = l2_evict_first_policy();
    constexpr int kScb = (FMT == MOE_W_Q8_0) ? 2 : 4;       // scale bytes per row
    constexpr int kScLanes = kScb;                           // lanes copying one block's 16 rows of scales
    // per-channel int8: panels of codes only, after the rows' fp32 scales (read again per panel)
    constexpr bool kPc = FMT == MOE_W_INT8PC;
    const int64_t stride = static_cast<int64_t>(rows) * (kPc ? 32 : 32 + kScb);
    const uint8_t* P = W + (kPc ? static_cast<int64_t>(rows) * 4 : 0) + static_cast<int64_t>(pb) * stride;
    const uint8_t* srcA = P + rowA * 32 + lane * 16;
    const uint8_t* srcB = P + rowB * 32 + lane * 16;
    const bool copies_scales = lane < 2 * kScLanes;
    const int sl = lane < kScLanes ? lane : lane - kScLanes;
    const uint8_t* srcS = (kPc ? W : P + static_cast<int64_t>(rows) * 32) + (lane < kScLanes ? rowA : rowB) * kScb +
                          sl * 16;
    const int64_t strideS = kPc ? 0 : stride;
    const uint32_t offS = 1024 + (lane < kScLanes ? 0 : 16 * kScb) + sl * 16;
    const uint32_t ring_addr = smem_addr(ring);
    const int n = pe - pb;
    auto issue = [&](int s) {
        const uint32_t slot = ring_addr + s * kSlotBytes;
        cp_async16_ef(slot + lane * 16, srcA, pol);
        cp_async16_ef(slot + 512 + lane * 16, srcB, pol);
        if (copies_scales) cp_async16(slot + offS, srcS);
        srcA += stride;
        srcB += stride;
        srcS += strideS;
    };
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
        if (s < n) issue(s);
        cp_async_commit();
    }
    between();   // block-wide: stage the activations while the first copies are in flight
    for (int i0 = 0; i0 < n; i0 += kStages) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            const int i = i0 + s;
            if (i < n) {
                cp_async_wait<kStages - 1>();
                __syncwarp();
                panel_mma<FMT>(ring + s * kSlotBytes, xs, ld, pb + i, nt, 0, acc, split, lo_off);
                __syncwarp();   // every lane is done with the slot before it is refilled
                if (i + kStages < n) issue(s);
                cp_async_commit();
            }
        }
    }
}


// Stage the f16 activations of `nt` tokens: x rows (gate.up) or h rows (down).  fp32
// sources also write the lo terms at + lo_off (bf16 sources are exact in one f16).
__device__ __forceinline__ void stage_x_f16(const ExpertArgs& a, const int4& si, int t0, int nt, __half* xs,
                                            int lo_off) {
    const int d4 = a.d / 4;
    for (int i = threadIdx.x; i < nt * d4; i += blockDim.x) {
        const int t = i / d4, c = (i % d4) * 4;
        const int64_t off = static_cast<int64_t>(slot_token(si, t0 + t, a.ws.perm, a.k)) * a.d + c;
        float4 v;
        if (a.xt == MOE_F32) {
            v = *reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + off);
        } else {
            const uint2 b = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + off);
            v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u),
                            __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u));
        }
        __half2 h01, h23, l01, l23;
        split_f16(v.x, v.y, h01, l01);
        split_f16(v.z, v.w, h23, l23);
        *reinterpret_cast<__half2*>(xs + t * a.d + c) = h01;
        *reinterpret_cast<__half2*>(xs + t * a.d + c + 2) = h23;
        if (a.xt == MOE_F32) {
            *reinterpret_cast<__half2*>(xs + lo_off + t * a.d + c) = l01;
            *reinterpret_cast<__half2*>(xs + lo_off + t * a.d + c + 2) = l23;
        }
    }
}

__device__ __forceinline__ void stage_h_f16(const ExpertArgs& a, int r0, int t0, int nt, __half* hs, int lo_off) {
    const int f4 = a.f / 4;
    const float4* src = reinterpret_cast<const float4*>(a.ws.h + static_cast<int64_t>(r0 + t0) * a.f);
    __half2* hi = reinterpret_cast<__half2*>(hs);
    __half2* lo = reinterpret_cast<__half2*>(hs + lo_off);
    for (int i = threadIdx.x; i < nt * f4; i += blockDim.x) {
        const float4 v = __ldcg(src + i);
        split_f16(v.x, v.y, hi[2 * i], lo[2 * i]);
        split_f16(v.z, v.w, hi[2 * i + 1], lo[2 * i + 1]);
    }
}

// Per-warp partial sums of a 32-row x 8-token tile into red[warp][blk][row][token].
__device__ __forceinline__ void store_partials(float* red, const float acc[2][4]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    float* r = red + warp * 256;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        r[blk * 128 + g * 8 + 2 * t] = acc[blk][0];
        r[blk * 128 + g * 8 + 2 * t + 1] = acc[blk][1];
        r[blk * 128 + (g + 8) * 8 + 2 * t] = acc[blk][2];
        r[blk * 128 + (g + 8) * 8 + 2 * t + 1] = acc[blk][3];
    }
}

// ------------------------------------------------------------------------------ gate.up
// grid: (f/16 tiles for SwiGLU: 16 gate rows and the 16 matching up rows; f/32 for ReLU^2:
// 32 up rows;  slot capacity); block 256 = 8 warps splitting the K panels.  Tokens of the
// slot's expert go 8 at a time through the MMA's N columns.
template <int FMT, int ACT>
__global__ void __launch_bounds__(256, 3) gate_up_gemv_kernel(ExpertArgs a) {
    pdl_wait();
    pdl_trigger();   // let the down kernel start filling its weight ring now
    const int slot = blockIdx.y;
    const int4 si = __ldcg(a.ws.slot_info + slot);
    const int e = si.x, r0 = si.y, cnt = si.z;
    if (cnt == 0) return;   // idle slot
    const int warp = threadIdx.x >> 5;
    extern __shared__ __align__(16) unsigned char dsm[];
    unsigned char* ring = dsm + warp * kStages * kSlotBytes;
    __half* xs = reinterpret_cast<__half*>(dsm + 8 * kStages * kSlotBytes);   // [tt][d]
    __shared__ float red[8 * 256];
    __shared__ uint32_t act_bits[8];
    // wpt warps share one tile's K panels; the CTA covers 8 / wpt consecutive tiles (with a
    // short K, each warp then streams a longer run of panels instead of a couple)
    const int wpt = a.gu_wpt, tpc = 8 / wpt;
    const int ntiles = (ACT == MOE_ACT_SWIGLU) ? a.f / 16 : a.f / 32;
    const int tile = blockIdx.x * tpc + warp / wpt, part = warp % wpt;
    const bool live = tile < ntiles;
    const int rowA = (ACT == MOE_ACT_SWIGLU) ? tile * 16 : tile * 32;
    const int rowB = (ACT == MOE_ACT_SWIGLU) ? a.f + tile * 16 : tile * 32 + 16;
    const uint8_t* W = a.w_gu + static_cast<int64_t>(e) * a.gu_bytes;
    const int npan = (FMT == MOE_W_NVFP4) ? a.d / 64 : a.d / 32;
    const int pb = live ? part * npan / wpt : 0, pe = live ? (part + 1) * npan / wpt : 0;
    if (threadIdx.x < 8) act_bits[threadIdx.x] = 0;
    if (threadIdx.x == 0) {
        if (a.prefetch_down) {   // this CTA's share of the expert's down matrix, into L2
            const int64_t share = ((a.dn_bytes + gridDim.x - 1) / gridDim.x + 127) / 128 * 128;
            const int64_t off = static_cast<int64_t>(blockIdx.x) * share;
            if (off < a.dn_bytes) {
                const int64_t n = min(share, a.dn_bytes - off);
                prefetch_l2(a.w_dn + static_cast<int64_t>(e) * a.dn_bytes + off, static_cast<uint32_t>(n));
            }
        }
        if (a.pf_bytes > 0) {   // this CTA's share of the caller's L2 hint (the next layer's router)
            const int64_t nct = static_cast<int64_t>(gridDim.x) * gridDim.y;
            const int64_t share = ((a.pf_bytes + nct - 1) / nct + 127) / 128 * 128;
            const int64_t off = (static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x) * share;
            if (off < a.pf_bytes) prefetch_l2(a.pf + off, static_cast<uint32_t>(min(share, a.pf_bytes - off)));
        }
    }
    const float ts = (FMT == MOE_W_NVFP4) ? a.gu_ts[e] : 1.0f;
    for (int t0 = 0; t0 < cnt; t0 += a.tt_gu) {
        const int nt = min(a.tt_gu, cnt - t0);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const bool split = a.xt == MOE_F32;
        const int lo_off = a.tt_gu * a.d;
        stream_panels_dense<FMT>(W, a.rows_gu, rowA, rowB, pb, pe, ring, xs, a.d, nt, acc, split, lo_off, [&] {
            stage_x_f16(a, si, t0, nt, xs, lo_off);
            __syncthreads();
        });
        store_partials(red, acc);
        __syncthreads();
        for (int it = threadIdx.x; it < tpc * 16 * 8; it += blockDim.x) {
            const int tl = it >> 7, row = (it >> 3) & 15, tok = it & 7;
            const int tt = blockIdx.x * tpc + tl;
            if (tok >= nt || tt >= ntiles) continue;
            float zA = 0.0f, zB = 0.0f;
            for (int w = tl * wpt; w < (tl + 1) * wpt; ++w) {   // the tile's warps in order
                zA += red[w * 256 + row * 8 + tok];
                zB += red[w * 256 + 128 + row * 8 + tok];
            }
            zA *= ts;
            zB *= ts;
            float* hrow = a.ws.h + static_cast<int64_t>(r0 + t0 + tok) * a.f;
            if (ACT == MOE_ACT_SWIGLU) {
                const float h = silu(zA) * zB;
                hrow[tt * 16 + row] = h;
                if (h != 0.0f) atomicOr(&act_bits[tl], 1u);
            } else {
                const float hA = zA > 0.0f ? zA * zA : 0.0f;
                const float hB = zB > 0.0f ? zB * zB : 0.0f;
                hrow[tt * 32 + row] = hA;
                hrow[tt * 32 + 16 + row] = hB;
                if (hA != 0.0f) atomicOr(&act_bits[tl], 1u);
                if (hB != 0.0f) atomicOr(&act_bits[tl], 2u);
            }
        }
        __syncthreads();   // red and xs are reused by the next token tile
    }
    if (threadIdx.x < tpc && act_bits[threadIdx.x]) {
        const int tt = blockIdx.x * tpc + threadIdx.x;
        const int g0 = (ACT == MOE_ACT_SWIGLU) ? tt : 2 * tt;
        const uint32_t bits = (ACT == MOE_ACT_SWIGLU) ? 1u : act_bits[threadIdx.x];
        atomicOr(a.ws.gmask + slot * a.gwords + g0 / 32, bits << (g0 % 32));
    }
}

// ------------------------------------------------------------------------------ fused combine
// pos / w of every pair in shared memory (the down kernels load them in their prologue).
constexpr int kMaxFusedPairs = 256;

__device__ __forceinline__ void preload_pairs(const ExpertArgs& a, int* spos, float* sw) {
    for (int p = threadIdx.x; p < a.P; p += blockDim.x) {
        spos[p] = __ldcg(a.ws.pos + p);
        sw[p] = __ldcg(a.ws.w + p);
    }
}

// Every CTA of the down grid (one per slot, idle slots included) arrives once per row tile;
// the last one of row tile [row0, row0+nrows) combines those rows for every token:
// out[t][r] = sum_{j<k} w[t][j] * y[pos(t,j)][r], in slot order.
__device__ __forceinline__ void combine_rows_if_last(const ExpertArgs& a, int tile, int row0, int nrows,
                                                     const int* spos, const float* sw, int nsplit = 1) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = (atomicAdd(a.ws.row_ctr + tile, 1) == static_cast<int>(gridDim.y) * nsplit - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int k = a.k;
    for (int it = threadIdx.x; it < a.T * nrows; it += blockDim.x) {
        const int t = it / nrows, r = row0 + it % nrows;
        float yj[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)     // every load of the item in flight at once
            if (j < k) yj[j] = __ldcg(a.ws.y + static_cast<int64_t>(spos[t * k + j]) * a.d + r);
        for (int z = 1; z < nsplit; ++z) {  // partial sums of the other group splits, in order
            const float* yz = a.ws.y + static_cast<int64_t>(z) * a.P * a.d;
#pragma unroll
            for (int j = 0; j < kMaxK; ++j)
                if (j < k) yj[j] += __ldcg(yz + static_cast<int64_t>(spos[t * k + j]) * a.d + r);
        }
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
            if (j < k) acc = fmaf(sw[t * k + j], yj[j], acc);
        a.out[static_cast<int64_t>(t) * a.d + r] = acc;
    }
    if (threadIdx.x == 0) a.ws.row_ctr[tile] = 0;
}

// ------------------------------------------------------------------------------ down, Q8_0
// Q8_0 down matrices [d][f] in K panels of 32 neurons.  A CTA = 32 output rows (two MMA
// blocks of 16); its 4 warps split the panels.  A panel holds neuron groups 2b and 2b+1;
// the 16 columns of an inactive group are neither copied nor used, and panels whose two
// groups are inactive are skipped.  grid: (d/32, slot capacity).
constexpr int kDnWarps = 4;

template <int FMT>   // Q8_0 or per-channel int8
__global__ void __launch_bounds__(kDnWarps * 32, 6) down_q8_gemv_kernel(ExpertArgs a) {
    const int slot = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    extern __shared__ __align__(16) unsigned char dsm[];
    unsigned char* ring = dsm + warp * kStages * kSlotBytes;
    __half* hs = reinterpret_cast<__half*>(dsm + kDnWarps * kStages * kSlotBytes);   // [tt][f] hi, then lo
    __shared__ uint32_t gm[64];
    __shared__ float red[kDnWarps * 256];
    __shared__ int spos[kMaxFusedPairs];
    __shared__ float sw[kMaxFusedPairs];
    // The slot records come from the routing kernel, which completed before the gate.up grid
    // this launch depends on could start: they and the weights may be read before waiting,
    // so the first panels stream in while gate.up is still running.
    const int4 si = __ldcg(a.ws.slot_info + slot);
    const int e = si.x, r0 = si.y, cnt = si.z;
    const int rt = blockIdx.x;
    const int npan = a.f / 32;
    const int pb = warp * npan / kDnWarps, pe = (warp + 1) * npan / kDnWarps;
    const uint8_t* W = a.w_dn + static_cast<int64_t>(e) * a.dn_bytes;
    const uint64_t pol = l2_evict_first_policy();
    const int rowA = rt * 32, rowB = rt * 32 + 16;
    const int npre = cnt > 0 ? min(kStages, pe - pb) : 0;
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
        if (s < npre) issue_panel_block<FMT>(smem_addr(ring + s * kSlotBytes), W, a.d, rowA, rowB, pb + s, pol, 0);
        cp_async_commit();
    }
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < a.gwords; i += blockDim.x) gm[i] = __ldcg(a.ws.gmask + slot * a.gwords + i);
    if (a.fuse_combine) preload_pairs(a, spos, sw);
    __syncthreads();
    // halves of inactive neuron groups: not copied (after the first panels) and not used
    auto skip_of = [&](int b) -> int {
        const int g = 2 * b;
        return (((gm[g >> 5] >> (g & 31)) & 1u) ? 0 : 1) | (((gm[(g + 1) >> 5] >> ((g + 1) & 31)) & 1u) ? 0 : 2);
    };
    const int lo_off = a.tt_dn * a.f;
    for (int t0 = 0; t0 < cnt; t0 += a.tt_dn) {
        const int nt = min(a.tt_dn, cnt - t0);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (t0 > 0) {   // later token tiles refill the ring
#pragma unroll
            for (int s = 0; s < kStages; ++s) {
                if (s < npre)
                    issue_panel_block<FMT>(smem_addr(ring + s * kSlotBytes), W, a.d, rowA, rowB, pb + s, pol,
                                                  skip_of(pb + s));
                cp_async_commit();
            }
        }
        stage_h_f16(a, r0, t0, nt, hs, lo_off);
        __syncthreads();
        for (int i = 0; pb + i < pe; ++i) {
            cp_async_wait<kStages - 1>();
            __syncwarp();
            const int s = i % kStages;
            panel_mma<FMT>(ring + s * kSlotBytes, hs, a.f, pb + i, nt, skip_of(pb + i), acc, true, lo_off);
            __syncwarp();
            const int bn = pb + i + kStages;
            if (bn < pe)
                issue_panel_block<FMT>(smem_addr(ring + s * kSlotBytes), W, a.d, rowA, rowB, bn, pol, skip_of(bn));
            cp_async_commit();
        }
        store_partials(red, acc);
        __syncthreads();
        for (int it = threadIdx.x; it < 32 * 8; it += blockDim.x) {
            const int blk = it >> 7, row = (it >> 3) & 15, tok = it & 7;
            if (tok >= nt) continue;
            float yv = 0.0f;
#pragma unroll
            for (int w = 0; w < kDnWarps; ++w) yv += red[w * 256 + blk * 128 + row * 8 + tok];
            a.ws.y[static_cast<int64_t>(r0 + t0 + tok) * a.d + rt * 32 + blk * 16 + row] = yv;
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    if (a.fuse_combine) combine_rows_if_last(a, rt, rt * 32, 32, spos, sw);
}

// ------------------------------------------------------------------------------ down, Q8_0, one token
// One token, SwiGLU (no group skips), k in {1, 2, 4, 8}: a CTA owns 16 output rows for every
// routed expert and combines them itself, so the expert outputs y never leave the CTA: no
// global round trip, atomic counter or last-CTA step.  Warp w works on slot w / wps (wps =
// 8 / k warps per slot, each a contiguous share of the K panels) through a ring of 16-row
// panel blocks (512 code bytes, then 16 fp16 scales).  grid: d/16 x 256 threads.
constexpr int kT1SlotBytes = 512 + 64;
constexpr int kT1Stages = 12;   // each warp walks a slot's whole K: a deeper ring than the other kernels

__global__ void __launch_bounds__(256, 2) down_q8_t1_kernel(ExpertArgs a, int wps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int row0 = blockIdx.x * 16;
    const int slot = warp / wps, part = warp % wps;
    extern __shared__ __align__(16) unsigned char dsm[];
    unsigned char* ring = dsm + warp * kT1Stages * kT1SlotBytes;
    __half* hs = reinterpret_cast<__half*>(dsm + 8 * kT1Stages * kT1SlotBytes);   // [k][f] hi, then lo
    __shared__ float red[8][16];
    __shared__ int s_pos[8];
    __shared__ float s_w[8];
    // Slot records come from the routing kernel, complete before the gate.up grid this
    // launch depends on started: the weights stream in while gate.up still runs.
    const int4 si = __ldcg(a.ws.slot_info + slot);
    const int e = si.x, hrow = si.y;
    const int npan = a.f / 32;
    const int pb = part * npan / wps, pe = (part + 1) * npan / wps;
    const int n = pe - pb;
    const int64_t stride = static_cast<int64_t>(a.d) * 34;
    const uint8_t* P = a.w_dn + static_cast<int64_t>(e) * a.dn_bytes + static_cast<int64_t>(pb) * stride;
    const uint8_t* srcC = P + static_cast<int64_t>(row0) * 32 + lane * 16;       // 16 rows x 32 codes = 32 x 16 B
    const uint8_t* srcS = P + static_cast<int64_t>(a.d) * 32 + row0 * 2 + lane * 16;   // 32 scale bytes, lanes 0-1
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t ring_addr = smem_addr(ring);
    auto issue = [&](int s) {
        const uint32_t sl = ring_addr + s * kT1SlotBytes;
        cp_async16_ef(sl + lane * 16, srcC, pol);
        if (lane < 2) cp_async16(sl + 512 + lane * 16, srcS);
        srcC += stride;
        srcS += stride;
    };
#pragma unroll
    for (int s = 0; s < kT1Stages; ++s) {
        if (s < n) issue(s);
        cp_async_commit();
    }
    pdl_wait();
    pdl_trigger();
    const int k = a.k;
    if (threadIdx.x < k) {   // the token's pairs: sorted row (= slot, one token) and weight
        s_pos[threadIdx.x] = __ldcg(a.ws.pos + threadIdx.x);
        s_w[threadIdx.x] = __ldcg(a.ws.w + threadIdx.x);
    }
    // h of the k pairs (sorted rows 0..k-1) as f16 hi + lo
    const int lo_off = k * a.f;
    {
        const float4* src = reinterpret_cast<const float4*>(a.ws.h);
        __half2* hi = reinterpret_cast<__half2*>(hs);
        __half2* lo = reinterpret_cast<__half2*>(hs + lo_off);
        for (int i = threadIdx.x; i < k * a.f / 4; i += blockDim.x) {
            const float4 v = __ldcg(src + i);
            split_f16(v.x, v.y, hi[2 * i], lo[2 * i]);
            split_f16(v.z, v.w, hi[2 * i + 1], lo[2 * i + 1]);
        }
    }
    __syncthreads();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const __half* xrow = hs + hrow * a.f;            // this slot's token (lane group g == 0)
    for (int i0 = 0; i0 < n; i0 += kT1Stages) {
#pragma unroll
        for (int s = 0; s < kT1Stages; ++s) {
            const int i = i0 + s;
            if (i < n) {
                cp_async_wait<kT1Stages - 1>();
                __syncwarp();
                const unsigned char* cb = ring + s * kT1SlotBytes;
                const int b = pb + i;
                uint4 xv = make_uint4(0, 0, 0, 0), xl = make_uint4(0, 0, 0, 0);
                if (g == 0) {
                    xv = *reinterpret_cast<const uint4*>(xrow + b * 32 + 8 * t);
                    xl = *reinterpret_cast<const uint4*>(xrow + lo_off + b * 32 + 8 * t);
                }
                const uint2 r0 = *reinterpret_cast<const uint2*>(cb + g * 32 + 8 * t);
                const uint2 r8 = *reinterpret_cast<const uint2*>(cb + (g + 8) * 32 + 8 * t);
                const unsigned short* sc = reinterpret_cast<const unsigned short*>(cb + 512);
                const float s0 = __half2float(__ushort_as_half(sc[g]));
                const float s8 = __half2float(__ushort_as_half(sc[g + 8]));
                uint32_t a0, a2, a1, a3, c0, c2, c1, c3;
                s8x4_to_f16x2x2(r0.x, a0, a2);
                s8x4_to_f16x2x2(r8.x, a1, a3);
                s8x4_to_f16x2x2(r0.y, c0, c2);
                s8x4_to_f16x2x2(r8.y, c1, c3);
                float dd[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(dd, a0, a1, a2, a3, xv.x, xv.y);
                mma16816(dd, c0, c1, c2, c3, xv.z, xv.w);
                mma16816(dd, a0, a1, a2, a3, xl.x, xl.y);
                mma16816(dd, c0, c1, c2, c3, xl.z, xl.w);
                acc[0] = fmaf(s0, dd[0], acc[0]);
                acc[2] = fmaf(s8, dd[2], acc[2]);
                __syncwarp();   // every lane is done with the slot before it is refilled
                if (i + kT1Stages < n) issue(s);
                cp_async_commit();
            }
        }
    }
    cp_async_wait<0>();
    // token column 0 of the accumulator: rows g (acc[0]) and g + 8 (acc[2]) on lanes t == 0
    if (t == 0) {
        red[warp][g] = acc[0];
        red[warp][g + 8] = acc[2];
    }
    __syncthreads();
    // y[slot][r]: the slot's warps in order; out[r] = sum over the token's pairs j in order
    if (threadIdx.x < 16) {
        const int r = threadIdx.x;
        float o = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int sj = s_pos[j];                  // sorted row of pair j = its slot (one token)
            float y = 0.0f;
            for (int q = 0; q < wps; ++q) y += red[sj * wps + q][r];
            o = fmaf(s_w[j], y, o);
        }
        a.out[row0 + r] = o;
    }
}

// ------------------------------------------------------------------------------ down, NVFP4
// NVFP4 down matrices in the neuron layout: per group of 16 neurons, each neuron's codes
// for all d rows (d/2 bytes), then the d scale bytes.  A CTA covers 256 rows (lane l:
// rows 8l .. 8l+7, 4 code bytes per neuron, 8 scale bytes); its 8 warps split the groups
// and meet in shared memory.  Inactive groups are not read at all.  grid: (d/256, slots,
// splits): with several splits (one token, fused combine) each CTA takes a share of the
// groups and writes a partial y; the combining CTA adds the splits in order.
// groups whose loads are in flight per warp (more costs registers, and with them the
// CTAs per SM that the split grid of the one-token case relies on)
template <int N>
constexpr int groups_in_flight() { return 2; }

template <int N>
__device__ __forceinline__ void dn_nv_tile(const ExpertArgs& a, const uint8_t* W, int rt, int gb, int ge,
                                           const uint32_t* gm, float* hs, int r0, int t0, int nt,
                                           float acc[N][8]) {
    const int d = a.d, f = a.f;
    const int lane = threadIdx.x & 31;
    const int64_t rec = 16 * (d / 2) + d;
    constexpr int kGif = groups_in_flight<N>();
    uint32_t codes[kGif][16];
    uint2 sc[kGif];
    int gid[kGif];
    int g = gb;
    // gather the next batch of active groups and issue their loads
    auto issue = [&]() {
        int n = 0;
        while (g < ge && n < kGif) {
            if ((gm[g >> 5] >> (g & 31)) & 1u) {
                gid[n] = g;
                ++n;
            }
            ++g;
        }
#pragma unroll
        for (int u = 0; u < kGif; ++u) {
            if (u < n) {
                const uint8_t* base = W + gid[u] * rec;
#pragma unroll
                for (int j = 0; j < 16; ++j) codes[u][j] = ldg_stream4(base + j * (d / 2) + rt * 128 + lane * 4);
                sc[u] = ldg_stream8(base + 16 * (d / 2) + rt * 256 + lane * 8);
            }
        }
        return n;
    };
    int n = issue();
    load_h_rows(a, r0, t0, nt, hs);
    __syncthreads();
    while (n > 0) {
#pragma unroll
        for (int u = 0; u < kGif; ++u) {
            if (u < n) {
                uint64_t part[N][4];   // rows (2by, 2by+1): one packed fmaf pair per code byte and token
#pragma unroll
                for (int t = 0; t < N; ++t)
#pragma unroll
                    for (int by = 0; by < 4; ++by) part[t][by] = 0;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    uint64_t hh[N];
#pragma unroll
                    for (int t = 0; t < N; ++t) {
                        const float hv = hs[t * f + 16 * gid[u] + j];
                        hh[t] = pack_f32x2(hv, hv);
                    }
#pragma unroll
                    for (int by = 0; by < 4; ++by) {
                        const float2 v = e2m1x2_to_f32x2((codes[u][j] >> (8 * by)) & 0xffu);   // rows 2by, 2by+1
                        const uint64_t vv = pack_f32x2(v.x, v.y);
#pragma unroll
                        for (int t = 0; t < N; ++t) fma_f32x2(part[t][by], vv, hh[t]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float sb = e4m3_to_f32(((r < 4 ? sc[u].x : sc[u].y) >> (8 * (r & 3))) & 0xffu);
#pragma unroll
                    for (int t = 0; t < N; ++t) {
                        const float2 pv = unpack_f32x2(part[t][r >> 1]);
                        acc[t][r] = fmaf(sb, (r & 1) ? pv.y : pv.x, acc[t][r]);
                    }
                }
            }
        }
        n = issue();
    }
}

template <int TT>
__global__ void __launch_bounds__(256, TT == 1 ? 3 : (TT == 2 ? 2 : 1)) down_nv_gemv_kernel(ExpertArgs a) {
    pdl_wait();
    pdl_trigger();
    const int slot = blockIdx.y;
    extern __shared__ __align__(16) float dyn[];
    float* hs = dyn;                                   // [TT][f]
    float* red = dyn + static_cast<size_t>(TT) * a.f;  // [8 warps][TT][256 rows]
    __shared__ uint32_t gm[64];
    __shared__ int spos[kMaxFusedPairs];
    __shared__ float sw[kMaxFusedPairs];
    const int4 si = __ldcg(a.ws.slot_info + slot);
    for (int i = threadIdx.x; i < a.gwords; i += blockDim.x) gm[i] = __ldcg(a.ws.gmask + slot * a.gwords + i);
    if (a.fuse_combine) preload_pairs(a, spos, sw);
    __syncthreads();
    const int e = si.x, r0 = si.y, cnt = si.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rt = blockIdx.x;
    const int ng = a.f / 16;
    const int z = blockIdx.z, nz = gridDim.z;
    const int zb = z * ng / nz, ze = (z + 1) * ng / nz;      // this split's groups
    const int gb = zb + warp * (ze - zb) / 8, ge = zb + (warp + 1) * (ze - zb) / 8;
    const uint8_t* W = a.w_dn + static_cast<int64_t>(e) * a.dn_bytes;
    const float ts = cnt > 0 ? a.dn_ts[e] : 0.0f;
    float* ydst = a.ws.y + static_cast<int64_t>(z) * a.P * a.d;
    for (int t0 = 0; t0 < cnt; t0 += TT) {
        const int nt = min(TT, cnt - t0);
#define MOE_DN_NV_CASE(NN)                                                                          \
    {                                                                                               \
        float acc[NN][8];                                                                           \
        _Pragma("unroll") for (int t = 0; t < NN; ++t) _Pragma("unroll") for (int r = 0; r < 8; ++r) \
            acc[t][r] = 0.0f;                                                                       \
        dn_nv_tile<NN>(a, W, rt, gb, ge, gm, hs, r0, t0, nt, acc);                                  \
        _Pragma("unroll") for (int t = 0; t < NN; ++t) {                                            \
            float* rr = red + (warp * TT + t) * 256 + lane * 8;                                     \
            *reinterpret_cast<float4*>(rr) = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]); \
            *reinterpret_cast<float4*>(rr + 4) = make_float4(acc[t][4], acc[t][5], acc[t][6], acc[t][7]); \
        }                                                                                           \
    }
        if (TT == 1 || nt == 1) MOE_DN_NV_CASE(1)
        else if (TT == 2 || nt == 2) MOE_DN_NV_CASE((TT < 2 ? TT : 2))
        else MOE_DN_NV_CASE((TT < 4 ? TT : 4))
#undef MOE_DN_NV_CASE
        __syncthreads();
        for (int it = threadIdx.x; it < nt * 256; it += blockDim.x) {
            const int t = it / 256, r = it % 256;
            float yv = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) yv += red[(w * TT + t) * 256 + r];
            ydst[static_cast<int64_t>(r0 + t0 + t) * a.d + rt * 256 + r] = yv * ts;
        }
        __syncthreads();
    }
    if (a.fuse_combine) combine_rows_if_last(a, rt, rt * 256, 256, spos, sw, nz);
}

// ------------------------------------------------------------------------------ down, NVFP4, tensor cores
// Two or more tokens: the neuron-layout matrices on mma.sync.  An E2M1 code times its E4M3
// block scale is exact in f16 (2 x 4 significant bits, magnitudes 2^-10 .. 2688), so each
// 16-neuron group is one K step of an m16n8k16 MMA with the scale folded into the weight
// fragment, the f32 accumulators run over all groups, and h rides as f16 hi + lo.
//   A warp covers 64 rows.  Lane (g, q) takes, of neurons 4q .. 4q+3, the code word of rows
// 8g .. 8g+7 (4 bytes each); MMA block mb (0..3) puts row 8g+2mb at M index g and row
// 8g+2mb+1 at g+8 (the low and high nibble of byte mb); K indices 2q, 2q+1 are neurons 4q,
// 4q+1 and 2q+8, 2q+9 are 4q+2, 4q+3, and the activations follow the same assignment.
//   A CTA covers 256 rows: warp w takes rows 64 (w & 3) .. and half w >> 2 of the slot's
// active groups; the two halves meet in shared memory in a fixed order.  Each warp streams
// its groups through a ring of cp.async stages: the 16 neurons' 32 code bytes at 32-byte
// slots n + n/4 (so that the four lanes of a quad read different banks), then 64 scale bytes.
// Tokens go in passes of 8 * NT (the h planes in shared memory); a slot's unused N tiles
// are skipped.  grid: (d/256, slots).
constexpr int kNvStages = 8;
constexpr int kNvStageBytes = 19 * 32 + 64;

__host__ __device__ constexpr int nv_h_ld(int f) { return f + ((16 - f % 64) + 64) % 64; }   // = 16 mod 64

size_t down_nv_mma_smem(int tt, int f) {
    const size_t h = static_cast<size_t>(2) * tt * nv_h_ld(f) * sizeof(__half);
    const size_t red = static_cast<size_t>(2) * tt * 257 * sizeof(float);
    return static_cast<size_t>(8) * kNvStages * kNvStageBytes + std::max(h, red) +
           static_cast<size_t>(f / 16) * sizeof(int);
}

template <int NT>
__global__ void __launch_bounds__(256, NT <= 2 ? 2 : 1) down_nv_mma_kernel(ExpertArgs a) {
    constexpr int TT = 8 * NT;
    const int slot = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int wq = warp & 3, half = warp >> 2;
    extern __shared__ __align__(16) unsigned char nsm[];
    unsigned char* ring = nsm + warp * kNvStages * kNvStageBytes;
    unsigned char* uni = nsm + 8 * kNvStages * kNvStageBytes;           // h planes, then the partial sums
    const int d = a.d, f = a.f, ng = f / 16, ld = nv_h_ld(f);
    __half* hs = reinterpret_cast<__half*>(uni);                       // [TT][ld] hi, then [TT][ld] lo
    float* red = reinterpret_cast<float*>(uni);                        // [2 halves][TT][257]
    const size_t h_bytes = static_cast<size_t>(2) * TT * ld * sizeof(__half);
    const size_t red_bytes = static_cast<size_t>(2) * TT * 257 * sizeof(float);
    const size_t uni_bytes = h_bytes > red_bytes ? h_bytes : red_bytes;
    int* glist = reinterpret_cast<int*>(uni + uni_bytes);               // active groups: half 0, then half 1
    __shared__ int s_na[2];
    pdl_wait();
    pdl_trigger();
    const int4 si = __ldcg(a.ws.slot_info + slot);
    const int e = si.x, r0 = si.y, cnt = si.z;
    if (cnt == 0) return;
    const int rt = blockIdx.x;
    const int R = rt * 256 + wq * 64;                                   // this warp's first row
    const uint8_t* W = a.w_dn + static_cast<int64_t>(e) * a.dn_bytes;
    const int64_t rec = 16 * static_cast<int64_t>(d / 2) + d;          // bytes of one group
    const float ts = a.dn_ts[e];
    const uint64_t pol = l2_evict_first_policy();
    // the active groups of each half, compacted by warps 0 and 4 (ballot + prefix count)
    if ((warp & 3) == 0) {
        const int gb = half ? ng / 2 : 0, ge = half ? ng : ng / 2;
        const uint32_t* gm = a.ws.gmask + static_cast<int64_t>(slot) * a.gwords;
        int n = 0;
        for (int c = gb; c < ge; c += 32) {
            const int gi = c + lane;
            const bool act = gi < ge && ((__ldcg(gm + (gi >> 5)) >> (gi & 31)) & 1u);
            const uint32_t bal = __ballot_sync(0xffffffffu, act);
            if (act) glist[gb + n + __popc(bal & ((1u << lane) - 1u))] = gi;
            n += __popc(bal);
        }
        if (lane == 0) s_na[half] = n;
    }
    __syncthreads();
    const int na = s_na[half];
    const int* mylist = glist + (half ? ng / 2 : 0);
    auto issue = [&](int st, int grp) {
        const uint32_t dst = smem_addr(ring + st * kNvStageBytes);
        const uint8_t* base = W + grp * rec;
        const int n = lane >> 1, h = lane & 1;
        cp_async16_ef(dst + (n + (n >> 2)) * 32 + h * 16, base + static_cast<int64_t>(n) * (d / 2) + R / 2 + h * 16,
                      pol);
        if (lane < 4) cp_async16(dst + 19 * 32 + lane * 16, base + 16 * static_cast<int64_t>(d / 2) + R + lane * 16);
    };
    for (int t0 = 0; t0 < cnt; t0 += TT) {
        const int nt = min(TT, cnt - t0);
#pragma unroll
        for (int s = 0; s < kNvStages; ++s) {
            if (s < na) issue(s, mylist[s]);
            cp_async_commit();
        }
        {   // h of this pass's tokens as f16 hi + lo planes
            const int f4 = f / 4;
            const float4* src = reinterpret_cast<const float4*>(a.ws.h + static_cast<int64_t>(r0 + t0) * f);
            for (int i = threadIdx.x; i < nt * f4; i += blockDim.x) {
                const int t = i / f4, c = (i % f4) * 4;
                const float4 v = __ldcg(src + i);
                __half2 h0, l0, h1, l1;
                split_f16(v.x, v.y, h0, l0);
                split_f16(v.z, v.w, h1, l1);
                __half2* hp = reinterpret_cast<__half2*>(hs + t * ld + c);
                __half2* lp = reinterpret_cast<__half2*>(hs + TT * ld + t * ld + c);
                hp[0] = h0;
                hp[1] = h1;
                lp[0] = l0;
                lp[1] = l1;
            }
        }
        __syncthreads();
        float acc[4][NT][4];
#pragma unroll
        for (int mb = 0; mb < 4; ++mb)
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[mb][n][0] = acc[mb][n][1] = acc[mb][n][2] = acc[mb][n][3] = 0.0f;
        for (int i = 0; i < na; ++i) {
            cp_async_wait<kNvStages - 1>();
            __syncwarp();
            const int st = i % kNvStages;
            const int grp = mylist[i];
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(ring + st * kNvStageBytes);
            const uint32_t c0 = sw[(4 * q + 0 + q) * 8 + g], c1 = sw[(4 * q + 1 + q) * 8 + g];
            const uint32_t c2 = sw[(4 * q + 2 + q) * 8 + g], c3 = sw[(4 * q + 3 + q) * 8 + g];
            const uint2 sc = *reinterpret_cast<const uint2*>(ring + st * kNvStageBytes + 19 * 32 + 8 * g);
            constexpr uint32_t m = 0x0f0f0f0fu;
            const uint32_t lo01 = (c0 & m) | ((c1 << 4) & ~m);   // byte b: row 8g+2b of neurons 4q | 4q+1
            const uint32_t hi01 = ((c0 >> 4) & m) | (c1 & ~m);   // row 8g+2b+1
            const uint32_t lo23 = (c2 & m) | ((c3 << 4) & ~m);
            const uint32_t hi23 = ((c2 >> 4) & m) | (c3 & ~m);
            // B fragments: token n*8+g, neurons 16 grp + 4q .. 4q+3 (hi and lo planes)
            uint2 bh[NT], bl[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const __half* hp = hs + (n * 8 + g) * ld + 16 * grp + 4 * q;
                bh[n] = *reinterpret_cast<const uint2*>(hp);
                bl[n] = *reinterpret_cast<const uint2*>(hp + TT * ld);
            }
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
                const uint32_t pair = ((mb < 2 ? sc.x : sc.y) >> (16 * (mb & 1))) & 0xffffu;   // rows 8g+2mb, +1
                uint32_t s2;
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2) : "h"(static_cast<uint16_t>(pair)));
                const __half2 sA = __low2half2(*reinterpret_cast<const __half2*>(&s2));
                const __half2 sB = __high2half2(*reinterpret_cast<const __half2*>(&s2));
                const int sh = 8 * mb;
                const uint32_t a0 = e2m1x2_scaled((lo01 >> sh) & 0xffu, sA);
                const uint32_t a1 = e2m1x2_scaled((hi01 >> sh) & 0xffu, sB);
                const uint32_t a2 = e2m1x2_scaled((lo23 >> sh) & 0xffu, sA);
                const uint32_t a3 = e2m1x2_scaled((hi23 >> sh) & 0xffu, sB);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    if (n * 8 < nt) {
                        mma16816(acc[mb][n], a0, a1, a2, a3, bh[n].x, bh[n].y);
                        mma16816(acc[mb][n], a0, a1, a2, a3, bl[n].x, bl[n].y);
                    }
                }
            }
            __syncwarp();
            if (i + kNvStages < na) issue(st, mylist[i + kNvStages]);
            cp_async_commit();
        }
        cp_async_wait<0>();
        __syncthreads();   // every warp is done with the h planes: the partial sums take their place
#pragma unroll
        for (int mb = 0; mb < 4; ++mb)
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int row = wq * 64 + 8 * g + 2 * mb, tok = n * 8 + 2 * q;
                float* rp = red + (half * TT + tok) * 257 + row;
                rp[0] = acc[mb][n][0];
                rp[257] = acc[mb][n][1];
                rp[1] = acc[mb][n][2];
                rp[258] = acc[mb][n][3];
            }
        __syncthreads();
        for (int it = threadIdx.x; it < nt * 256; it += blockDim.x) {
            const int t = it >> 8, r = it & 255;
            const float v = red[t * 257 + r] + red[(TT + t) * 257 + r];
            a.ws.y[static_cast<int64_t>(r0 + t0 + t) * d + rt * 256 + r] = v * ts;
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------------------ combine
// out[t] = sum_{j<k} w[t][j] * y[pos(t,j)], in slot order.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ w, const int32_t* __restrict__ pos,
                                                       const float* __restrict__ y, int k, int d,
                                                       float* __restrict__ out) {
    pdl_wait();
    const int t = blockIdx.y;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (c >= d) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int r = pos[t * k + j];
        const float wt = w[t * k + j];
        const float4 v = *reinterpret_cast<const float4*>(y + static_cast<int64_t>(r) * d + c);
        acc.x = fmaf(wt, v.x, acc.x);
        acc.y = fmaf(wt, v.y, acc.y);
        acc.z = fmaf(wt, v.z, acc.z);
        acc.w = fmaf(wt, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + static_cast<int64_t>(t) * d + c) = acc;
}

// ------------------------------------------------------------------------------ rmsnorm glue
// One CTA per token: every thread loads its elements first, then a fixed-order reduction.
constexpr int kNormMaxPerThread = 32;

__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ x, int d, float eps,
                                                            uint16_t* __restrict__ xo) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const float* xr = x + static_cast<int64_t>(t) * d;
    float v[kNormMaxPerThread];
    float ss = 0.0f;
    for (int base = 0; base < d; base += 256 * kNormMaxPerThread) {
#pragma unroll
        for (int u = 0; u < kNormMaxPerThread; ++u) {
            const int i = base + u * 256 + threadIdx.x;
            v[u] = (i < d) ? xr[i] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kNormMaxPerThread; ++u) ss = fmaf(v[u], v[u], ss);
    }
    ss = warp_sum(ss);
    __shared__ float wsum[8];
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += wsum[i];
    const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
    if (d <= 256 * kNormMaxPerThread) {
#pragma unroll
        for (int u = 0; u < kNormMaxPerThread; ++u) {
            const int i = u * 256 + threadIdx.x;
            if (i < d) xo[static_cast<int64_t>(t) * d + i] = __bfloat16_as_ushort(__float2bfloat16_rn(v[u] * inv));
        }
    } else {
        for (int i = threadIdx.x; i < d; i += 256)
            xo[static_cast<int64_t>(t) * d + i] = __bfloat16_as_ushort(__float2bfloat16_rn(xr[i] * inv));
    }
}

// ------------------------------------------------------------------------------ launchers
// Raise the kernel's dynamic shared-memory limit and ask for the largest shared-memory
// carveout, so that as many CTAs fit per SM as registers allow.
template <typename K>
static cudaError_t allow_smem(K kernel, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

template <int FMT, int ACT>
static cudaError_t gu_launch(const ExpertArgs& a, dim3 grid, size_t smem, cudaStream_t s, bool configure) {
    if (configure) return allow_smem(gate_up_gemv_kernel<FMT, ACT>, 200 * 1024);
    return launch_pdl(gate_up_gemv_kernel<FMT, ACT>, grid, dim3(256), smem, s, a);
}

static cudaError_t gu_dispatch(const ExpertArgs& a, int wfmt, int act, dim3 grid, size_t smem, cudaStream_t s,
                               bool configure) {
    if (wfmt == MOE_W_Q8_0 && act == MOE_ACT_SWIGLU) return gu_launch<MOE_W_Q8_0, MOE_ACT_SWIGLU>(a, grid, smem, s, configure);
    if (wfmt == MOE_W_Q8_0) return gu_launch<MOE_W_Q8_0, MOE_ACT_RELU2>(a, grid, smem, s, configure);
    if (wfmt == MOE_W_INT8PC && act == MOE_ACT_SWIGLU)
        return gu_launch<MOE_W_INT8PC, MOE_ACT_SWIGLU>(a, grid, smem, s, configure);
    if (wfmt == MOE_W_INT8PC) return gu_launch<MOE_W_INT8PC, MOE_ACT_RELU2>(a, grid, smem, s, configure);
    if (act == MOE_ACT_SWIGLU) return gu_launch<MOE_W_NVFP4, MOE_ACT_SWIGLU>(a, grid, smem, s, configure);
    return gu_launch<MOE_W_NVFP4, MOE_ACT_RELU2>(a, grid, smem, s, configure);
}

template <int TT>
static cudaError_t dn_nv_launch(const ExpertArgs& a, int slot_cap, size_t smem, cudaStream_t s, bool configure) {
    if (configure) return allow_smem(down_nv_gemv_kernel<TT>, 200 * 1024);
    return launch_pdl(down_nv_gemv_kernel<TT>, dim3(a.d / 256, slot_cap, a.nv_split), dim3(256), smem, s, a);
}

template <int NT>
static cudaError_t nv_mma_launch(const ExpertArgs& a, int slot_cap, cudaStream_t s, bool configure) {
    if (configure) return allow_smem(down_nv_mma_kernel<NT>, 200 * 1024);
    return launch_pdl(down_nv_mma_kernel<NT>, dim3(a.d / 256, slot_cap), dim3(256), down_nv_mma_smem(8 * NT, a.f), s,
                      a);
}

static cudaError_t dn_dispatch(const ExpertArgs& a, int wfmt, int slot_cap, size_t smem, cudaStream_t s,
                               bool configure) {
    if (wfmt == MOE_W_Q8_0) {
        if (configure) return allow_smem(down_q8_gemv_kernel<MOE_W_Q8_0>, 200 * 1024);
        return launch_pdl(down_q8_gemv_kernel<MOE_W_Q8_0>, dim3(a.d / 32, slot_cap), dim3(kDnWarps * 32), smem, s, a);
    }
    if (wfmt == MOE_W_INT8PC) {
        if (configure) return allow_smem(down_q8_gemv_kernel<MOE_W_INT8PC>, 200 * 1024);
        return launch_pdl(down_q8_gemv_kernel<MOE_W_INT8PC>, dim3(a.d / 32, slot_cap), dim3(kDnWarps * 32), smem, s,
                          a);
    }
    if (a.nv_mma || configure) {
        cudaError_t e = cudaSuccess;
        switch (a.tt_dn) {
            case 32: e = nv_mma_launch<4>(a, slot_cap, s, configure); break;
            case 16: e = nv_mma_launch<2>(a, slot_cap, s, configure); break;
            default: e = nv_mma_launch<1>(a, slot_cap, s, configure); break;
        }
        if (!configure || e != cudaSuccess) return e;
    }
    switch (a.tt_dn) {
        case 1: return dn_nv_launch<1>(a, slot_cap, smem, s, configure);
        case 2: return dn_nv_launch<2>(a, slot_cap, smem, s, configure);
        default: return dn_nv_launch<4>(a, slot_cap, smem, s, configure);
    }
}

// Raise the dynamic shared-memory limit of every expert-kernel instantiation (once per
// device).
cudaError_t configure_gemv_kernels() {
    ExpertArgs a{};
    const int wf[3] = {MOE_W_Q8_0, MOE_W_NVFP4, MOE_W_INT8PC};
    const int ac[2] = {MOE_ACT_SWIGLU, MOE_ACT_RELU2};
    for (int w : wf)
        for (int c : ac) {
            cudaError_t e = gu_dispatch(a, w, c, dim3(1), 0, nullptr, true);
            if (e != cudaSuccess) return e;
        }
    cudaError_t e0 = allow_smem(down_q8_t1_kernel, 200 * 1024);
    if (e0 != cudaSuccess) return e0;
    const int tts[6] = {1, 2, 4, 8, 16, 32};
    for (int tt : tts) {
        a.tt_dn = tt;
        for (int w : wf) {
            cudaError_t e = dn_dispatch(a, w, 1, 0, nullptr, true);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_gate_up_gemv(const ExpertArgs& a, int wfmt, int act, int slot_cap, cudaStream_t s) {
    const int ntiles = (act == MOE_ACT_SWIGLU) ? a.f / 16 : a.f / 32;
    const int tpc = 8 / a.gu_wpt;                       // tiles per CTA
    const int ctas_x = (ntiles + tpc - 1) / tpc;
    const size_t smem = static_cast<size_t>(8) * kStages * kSlotBytes +
                        static_cast<size_t>(a.tt_gu) * a.d * 2 * (a.xt == MOE_F32 ? 2 : 1);
    return gu_dispatch(a, wfmt, act, dim3(ctas_x, slot_cap), smem, s, false);
}

size_t down_gemv_smem(int wfmt, int tt_dn, int f) {
    if (wfmt == MOE_W_NVFP4) {
        const int t4 = tt_dn < 4 ? tt_dn : 4;
        return static_cast<size_t>(t4) * f * sizeof(float) + static_cast<size_t>(8) * t4 * 256 * sizeof(float);
    }
    return static_cast<size_t>(kDnWarps) * kStages * kSlotBytes + static_cast<size_t>(tt_dn) * f * 2 * 2;
}

size_t down_t1_smem(int k, int f) {
    return static_cast<size_t>(8) * kT1Stages * kT1SlotBytes + static_cast<size_t>(k) * f * 2 * 2;
}

cudaError_t launch_down_q8_t1(const ExpertArgs& a, cudaStream_t s) {
    const int wps = 8 / a.k;
    return launch_pdl(down_q8_t1_kernel, dim3(a.d / 16), dim3(256), down_t1_smem(a.k, a.f), s, a, wps);
}

cudaError_t launch_down_gemv(const ExpertArgs& a, int wfmt, int slot_cap, cudaStream_t s) {
    return dn_dispatch(a, wfmt, slot_cap, down_gemv_smem(wfmt, a.tt_dn, a.f), s, false);
}

cudaError_t launch_combine(const float* w, const int32_t* pos, const float* y, int64_t T, int k, int64_t d,
                           float* out, cudaStream_t s) {
    const int64_t cols4 = d / 4;
    const dim3 grid(static_cast<unsigned>((cols4 + 255) / 256), static_cast<unsigned>(T));
    return launch_pdl(combine_kernel, grid, dim3(256), 0, s, w, pos, y, k, static_cast<int>(d), out);
}

cudaError_t launch_rmsnorm_bf16(const float* x, int64_t T, int64_t d, float eps, uint16_t* xo, cudaStream_t s) {
    return launch_pdl(rmsnorm_bf16_kernel, dim3(static_cast<unsigned>(T)), dim3(256), 0, s, x, static_cast<int>(d),
                      eps, xo);
}

}  // namespace moe
