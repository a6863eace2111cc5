// decode.cu -- routed MoE layers for ONE token as a single persistent kernel: one layer
// (moe_layer_forward) or a whole stack of layers glued by the RMS-norm (moe_stack_forward).
//
// The same layer as route.cu + gemv.cu (router, top-k, softmax over the selected logits,
// gate.up with the activation, down projection, fixed-order combine), for the case that
// decides decode speed: one token, where the layer moves only the routed experts' weights
// (a few tens of MB) and the separate launches' start-up, ramp and tail cost more than the
// bytes.  Expert formats: Q8_0 or per-channel int8 with SwiGLU, and NVFP4 with ReLU^2
// (gateless latent experts) or SwiGLU.  Sources of the computation:
//   router / top-k / softmax: "Squeezing a 26B MoE onto the cheapest Inferentia instance"
//     (128 experts, top-8 per token), with the canonical fp32 summation order of the oracle;
//   gate.up + SwiGLU: "Running Gemma 4 26B at 5 tokens/s on a 13-year-old Xeon", sections
//     "A three-step fix" / "Runtime graph fallback" (fused [n_embd, 2*n_ff, n_experts]
//     tensor, gate rows first, then SiLU(gate)*up);
//   ReLU^2 experts and the down projection over 16-neuron groups that hold a non-zero
//     activation: "Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU", section
//     "How the engine works", step 4;
//   combine: the same page, section "How we check correctness" (per-(token, expert) results
//     summed in a fixed order, no atomics on the values).
//
// One CTA per SM (a cooperative launch: every CTA is resident, so the grid barriers below
// cannot wait on a CTA that never runs), 16 warps each.  Per layer:
//   R  CTA c < E/epc computes the logits of experts [c*epc, (c+1)*epc) in the canonical
//      order (256 fma chains i = l (mod 256), then the halving tree); its slice of the
//      router weights is copied into shared memory before the kernel waits for the
//      previous one (in a stack: while the previous layer finishes).  Barrier.  With up to
//      256 experts every CTA then ranks all E logits itself (top-k, lower index on ties;
//      2 to 8 lanes per expert); with more, the routing CTAs rank their own experts and
//      publish the winners behind one more barrier (a separate instantiation of the kernel).
//      The softmax over the selected logits and the routing record follow the first gate.up
//      requests, which need only the selection.
//   G  gate.up: the panel products of all k experts (items of 16 gate + 16 up rows, or 32
//      rows for ReLU^2) are one flattened range split evenly over the warps of the grid, so
//      every warp streams the same number of panels (within one) whatever the shapes.  A
//      CTA's warps cover a contiguous stretch of items: their partials meet in shared
//      memory and the CTA writes one record per item it touched.  Q8_0: each CTA also asks
//      L2 for its share of the routed experts' down matrices.  Barrier.
//   H  each CTA sums the records of the slots its down units read (in CTA order) and applies
//      the activation into its own copy of h (NVFP4: and flags the 16-neuron groups that
//      hold a non-zero h).
//   D  down, flattened the same way: Q8_0 units (slot, 32-row tile, 32-neuron panel), one
//      record per warp and item (the first ring stages are requested before H); NVFP4
//      units (slot, 256-row tile, 16-neuron group), only flagged groups read, one record
//      per CTA and item.  Barrier.
//   C  rows are combined by CTA (row chunk) mod G: y per slot (records in order), then the
//      pairs in order j: out[r] = sum_j w_j * y_{slot(j)}[r].
//   N  (stacks) barrier; every CTA computes the next layer's input, the RMS-norm of out in
//      the reduction order of the stand-alone norm kernel.
// Every per-warp quantity that depends only on the shapes is worked out before the kernel
// waits for the previous one.  All waits are bounded (about one second, then device error 2
// and the kernel goes on), so a barrier can never hang the GPU.  Results are bitwise
// reproducible run to run: every sum has a fixed order.
#include "gemv_core.cuh"

namespace moe {

namespace {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDevErrTimeout = 2;
constexpr long long kWaitLimitNs = 1000000000ll;   // bounded waits: one second
constexpr size_t kRingBytes = static_cast<size_t>(kDecWarps) * kStages * kSlotBytes;
constexpr int kLocalRankMaxE = 256;   // up to this many experts every CTA ranks all logits itself
// Routing modes of the kernel (a template parameter: each kernel holds only its own code)
constexpr int kRouteLocal = 0;      // router, then every CTA ranks all E <= 256 logits
constexpr int kRouteWide = 1;       // router, then the routing CTAs rank their own experts (E > 256)
constexpr int kRouteSupplied = 2;   // the caller's idx / w (one layer): no router, no selection

__device__ __forceinline__ long long globaltimer() {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier over a monotonically growing counter (target = n * gridDim.x for the
// n-th barrier of a call).  Bounded: a wait that passes `limit_ns` records device error 2 and
// raises the counter past every target of the call, so that no CTA waits again: the kernel
// then runs to its end at once.  The data behind a barrier that was given up on may be stale;
// every index the kernel reads from the workspace is clamped to its range, so the stale values
// can make the output wrong (error 2 declares it invalid) but cannot make an access leave its
// buffer.  The normal path costs nothing extra: no flag is read outside the spin.
constexpr int32_t kBarrierGiveUp = 1 << 30;   // above every target: 64 layers x 5 barriers x 256 CTAs

__device__ __forceinline__ void grid_barrier(int32_t* ctr, int target, int32_t* err, long long limit_ns) {
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: the CTA's writes (ordered before this by the barrier above) are visible to
        // every CTA that acquires the counter at or past the target
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(ctr) : "memory");
        if (ld_acquire(ctr) < target) {
            const long long t0 = globaltimer();
            while (ld_acquire(ctr) < target) {
                if (globaltimer() - t0 > limit_ns) {
                    set_error(err, kDevErrTimeout);
                    atomicMax(ctr, kBarrierGiveUp);
                    break;
                }
            }
        }
    }
    __syncthreads();
}


// An even split of U units over W warps: warp w owns [begin(w), begin(w+1)).  The host
// admits only shapes with (U + 1) * W < 2^32, so the arithmetic stays 32-bit.
__device__ __forceinline__ uint32_t split_begin(uint32_t U, uint32_t W, uint32_t w) { return w * U / W; }
// The warp that owns unit u: the largest w with begin(w) <= u.
__device__ __forceinline__ uint32_t split_owner(uint32_t U, uint32_t W, uint32_t u) { return ((u + 1) * W + U - 1) / U - 1; }
// Warps that own units of item i (units [i * npan, (i + 1) * npan)).
__device__ __forceinline__ int item_contributors(uint32_t U, uint32_t W, uint32_t npan, uint32_t i) {
    return static_cast<int>(split_owner(U, W, (i + 1) * npan - 1) - split_owner(U, W, i * npan)) + 1;
}

__device__ __forceinline__ bool beats(float va, int ea, float vb, int eb) { return va > vb || (va == vb && ea < eb); }

// Selection for many experts, by a routing CTA (all of its threads): each of its own epc
// experts is ranked among all E logits (lg) by 512/epc threads, and an expert of rank < k is
// published at its rank.  Only the kernels for more than 256 experts hold this code (a
// template parameter): the extra code, and even an out-of-line call, measurably slowed the
// kernels of the common shapes.
__device__ __forceinline__ void rank_own_experts(const float* lg, int* cnt, int E, int k, int epc, int c, int32_t* sel,
                                              float* selv) {
    const int tid = threadIdx.x, warp = tid >> 5;
    const int tpx = kDecThreads / epc;
    const int j = tid / tpx, part = tid % tpx;
    const int e = c * epc + j;
    const float v = lg[e];
    int r = 0;
#pragma unroll 1
    for (int o = part * E / tpx; o < (part + 1) * E / tpx; ++o) r += beats(lg[o], o, v, e);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
    if ((tid & 31) == 0) cnt[warp] = r;
    __syncthreads();
    if (part == 0) {
        int rank = 0;
        for (int w = j * tpx / 32; w < (j + 1) * tpx / 32; ++w) rank += cnt[w];
        if (rank < k) {
            sel[rank] = e;
            selv[rank] = v;
        }
    }
}

// A warp's share of one phase: units [u0, u0 + n) starting at panel b0 of item item0, whose
// first record goes to contributor slot c0 of that item (later items: slot 0).
struct WarpRange {
    int n, item0, b0, c0;
};

__device__ __forceinline__ WarpRange warp_range(uint32_t U, uint32_t W, uint32_t npan, uint32_t gw) {
    WarpRange r{0, 0, 0, 0};
    if (gw >= W) return r;
    const uint32_t u0 = split_begin(U, W, gw), u1 = split_begin(U, W, gw + 1);
    r.n = static_cast<int>(u1 - u0);
    r.item0 = static_cast<int>(u0 / npan);
    r.b0 = static_cast<int>(u0 % npan);
    r.c0 = static_cast<int>(gw - split_owner(U, W, static_cast<uint32_t>(r.item0) * npan));
    return r;
}

}  // namespace

// Shared-memory plan (dynamic): [ring | B | C | P]; B at the constant offset kRingBytes, the
// offsets of C and P computed on the host
//   ring : per-warp rings of panel blocks (16 x 6 x 1152 B), gate.up then down (Q8_0); during
//          routing, the CTA's router-weight slice [d][epc] and the tree buffer [epc][256];
//          NVFP4 down: the CTA's per-warp partials [items][16 warps][256]
//   B    : x as fp32 [d] (routing), then h: Q8_0 f16 hi [k][f] + lo [k][f], NVFP4 fp32 for the
//          CTA's slots [slots][f]
//   C    : x as f16 hi [d] (+ lo [d] for fp32 inputs) (gate.up)
//   P    : the per-warp gate.up partials of the CTA's items [cta_items][16 warps][32]
size_t decode_smem_plan(int wfmt, int d, int f, int k, int xt, int cta_items, int cta_slots, int* off_c, int* off_p) {
    const size_t xb = static_cast<size_t>(d) * 4;
    const size_t hb = (wfmt != MOE_W_NVFP4) ? static_cast<size_t>(k) * f * 4 : static_cast<size_t>(cta_slots) * f * 4;
    const size_t b = xb > hb ? xb : hb;
    const size_t cbytes = static_cast<size_t>(d) * 2 * (xt == MOE_F32 ? 2 : 1);
    const size_t pb = static_cast<size_t>(cta_items) * kDecWarps * 32 * sizeof(float);
    if (off_c) *off_c = static_cast<int>(kRingBytes + b);
    if (off_p) *off_p = static_cast<int>(kRingBytes + b + cbytes);
    return kRingBytes + b + cbytes + pb;
}

size_t decode_ring_bytes() { return kRingBytes; }

template <int FMT, int ACT, int ROUTE, bool AQ>
__global__ void __launch_bounds__(kDecThreads, 1) decode_layer_kernel(DecodeArgs a) {
    // Q8_0 or per-channel int8 with SwiGLU (32-column int8 panels with block or row scales),
    // or NVFP4 with ReLU^2 (gateless latent experts) or SwiGLU
    constexpr bool kQ8 = FMT == MOE_W_Q8_0 || FMT == MOE_W_INT8PC;
    // AQ (Q8_0 only): the experts read x and h through the Q8_0 activation coder (blocks of 32,
    // the values the codes stand for, carried as f16 hi + lo); the router reads x as it is
    static_assert(!AQ || (FMT == MOE_W_Q8_0 && ACT == MOE_ACT_SWIGLU), "coded activations: Q8_0 SwiGLU");
    constexpr bool kSupplied = ROUTE == kRouteSupplied;
    constexpr bool kSwiglu = ACT == MOE_ACT_SWIGLU;
    constexpr int kNeur = kSwiglu ? 16 : 32;   // neurons per gate.up item (16 gate + 16 up rows, or 32 rows)
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ __align__(16) float slog[kMaxE];   // logits; later the contributor counts of the gate.up items
    __shared__ int s_sel[kMaxK];     // expert of selection slot j (larger logit first)
    __shared__ float s_val[kMaxK];   // its logit
    __shared__ int s_e[kMaxK];       // expert of sorted slot s (increasing expert index)
    __shared__ int s_pos[kMaxK];     // sorted slot of pair j
    __shared__ float s_w[kMaxK];     // combine weight of pair j
    __shared__ int s_cnt[kDecWarps]; // per-warp counts (ranking over many experts)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the grid barriers' wait limit: the workspace's limit word when set (tests), else a second
    const long long wait_lim = *reinterpret_cast<const volatile long long*>(a.bar + kWaitLimitWord);
    const long long wait_ns = wait_lim > 0 ? wait_lim : kWaitLimitNs;
    const int G = gridDim.x, c = blockIdx.x;
    const int d = a.d, f = a.f, E = a.E, k = a.k;
    const uint32_t gw = static_cast<uint32_t>(c * kDecWarps + warp);   // warp index in the grid
    unsigned char* ring = dsm;
    // region B starts at a constant offset: its accesses (h in the down phase above all) use
    // immediate shared-memory addresses, measurably faster than a base passed in the arguments
    float* xf = reinterpret_cast<float*>(dsm + kRingBytes);
    __half* xh = reinterpret_cast<__half*>(dsm + a.off_c);
    const bool split = a.xt == MOE_F32 || AQ;   // x for the experts as f16 hi + lo (fp32 input, or coded)
    // the two streaming phases: items, panels per item, units
    // gate.up: items (slot, tile of kNeur neurons), panels of 32 (Q8_0) or 64 (NVFP4) columns
    const int nt_g = f / kNeur, npan_g = kQ8 ? d / 32 : d / 64;
    // down: Q8_0 items (slot, 32-row tile), units 32-neuron panels; NVFP4 items (slot, 256-row
    // tile), units 16-neuron groups of the neuron-contiguous layout
    const int npan_d = kQ8 ? f / 32 : f / 16;
    const int nrt = kQ8 ? d / 32 : d / 256;
    const uint32_t items_g = static_cast<uint32_t>(k * nt_g), items_d = static_cast<uint32_t>(nrt * k);
    const uint32_t U_g = items_g * npan_g, U_d = items_d * npan_d;
    // shape-only bookkeeping, done before waiting for the previous kernel
    const WarpRange rg = warp_range(U_g, a.warps_g, npan_g, gw);
    const WarpRange rd = warp_range(U_d, a.warps_d, npan_d, gw);

    // ---------------------------------------------------------------- R: router logits
    const int epc = a.epc;
    const bool router = c < E / epc;
    float* wsl = reinterpret_cast<float*>(ring);   // [d][epc]
    float* red = wsl + d * epc;                     // [epc][256]
    // this CTA's slice of a layer's router weights, copied asynchronously into the ring region
    auto request_router = [&](const float* W) {
        if (kSupplied || !router) return;
        const float* src = W + c * epc;
        const uint32_t wb = smem_addr(wsl);
        for (int it = tid; it < d * epc; it += kDecThreads) {
            const int i = it / epc, e = it % epc;
            cp_async4(wb + static_cast<uint32_t>(it) * 4, src + static_cast<int64_t>(i) * E + e);
        }
        cp_async_commit();
    };
    request_router(a.lp[0].W);   // does not depend on the previous kernel: before waiting for it
    pdl_wait();
    for (int i = tid; i < d / 4; i += kDecThreads) {   // (whole warps: d / 4 is a multiple of 64)
        float4 v;
        if (AQ ? a.xt == MOE_F32 : split) {   // (split: an fp32 input, unless coded)
            v = __ldcg(reinterpret_cast<const float4*>(a.x) + i);
        } else {
            const uint2 b = __ldcg(reinterpret_cast<const uint2*>(a.x) + i);
            v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u), __uint_as_float(b.y << 16),
                            __uint_as_float(b.y & 0xffff0000u));
        }
        reinterpret_cast<float4*>(xf)[i] = v;
        if constexpr (AQ) {   // the experts' x: each block of 32 (8 threads) through the coder
            uint32_t mb = max(max(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y))),
                              max(__float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w))));
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, m));
            const float amax = __uint_as_float(mb);
            v = make_float4(q8_0_coded_value(v.x, amax), q8_0_coded_value(v.y, amax), q8_0_coded_value(v.z, amax),
                            q8_0_coded_value(v.w, amax));
        }
        __half2 h01, h23, l01, l23;
        split_f16(v.x, v.y, h01, l01);
        split_f16(v.z, v.w, h23, l23);
        reinterpret_cast<__half2*>(xh)[2 * i] = h01;
        reinterpret_cast<__half2*>(xh)[2 * i + 1] = h23;
        if (split) {
            reinterpret_cast<__half2*>(xh + d)[2 * i] = l01;
            reinterpret_cast<__half2*>(xh + d)[2 * i + 1] = l23;
        }
    }
    int nbar = 0;   // grid barriers passed (the counter target of the next is (nbar + 1) * G)
    for (int l = 0; l < a.n_layers; ++l) {
        const DecodeLayerPtrs P = a.lp[l];
        const bool split_l = (l == 0 && split) || AQ;   // later layers read bf16 inputs: one f16 term, unless coded
        cp_async_wait<0>();
        __syncthreads();
        if (!kSupplied && router) {
            if (tid < kRouterPartials) {   // chain l: fmaf over i = l, l + 256, ... in increasing i
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
                const int nchain = d / kRouterPartials;
                for (int m = 0; m < nchain; ++m) {
                    const int i = tid + m * kRouterPartials;
                    const float xv = xf[i];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e < epc) acc[e] = fmaf(xv, wsl[i * epc + e], acc[e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e < epc) red[e * kRouterPartials + tid] = acc[e];
            }
            __syncthreads();
            for (int h = kRouterPartials / 2; h >= 32; h >>= 1) {   // s_l += s_{l+h}, h = 128, 64, 32
                for (int it = tid; it < epc * h; it += kDecThreads) {
                    const int e = it / h, l = it % h;
                    red[e * kRouterPartials + l] = red[e * kRouterPartials + l] + red[e * kRouterPartials + l + h];
                }
                __syncthreads();
            }
            if (warp < epc) {   // h = 16 .. 1 across the lanes; lane 0 ends with s_0
                float v = red[warp * kRouterPartials + lane];
#pragma unroll
                for (int h = 16; h >= 1; h >>= 1) v = v + __shfl_down_sync(0xffffffffu, v, h);
                if (lane == 0) a.ws.logits[c * epc + warp] = v;
            }
        }
        if constexpr (!kSupplied) grid_barrier(a.bar, ++nbar * G, a.ws.err, wait_ns);
        if (l == 0) pdl_trigger();   // every CTA is resident: the next kernel may be scheduled

        // ---------------------------------------------------------------- R: top-k, weights, slots
        // Up to 256 experts every CTA ranks all the logits itself.  With more, the O(E^2)
        // comparisons would cost a CTA microseconds: each routing CTA ranks only its own
        // experts among all E logits and publishes the winners, and after one more grid barrier
        // every CTA reads the k winners.
        constexpr bool wide = ROUTE == kRouteWide;   // launched exactly when E > kLocalRankMaxE
        if (!kSupplied && (!wide || router))
            for (int e = tid; e < E; e += kDecThreads) slog[e] = __ldcg(a.ws.logits + e);
        // gate.up items this CTA's warps touch, and their per-warp partials [items][16 warps][32]
        const uint32_t wc0 = min(static_cast<uint32_t>(c * kDecWarps), static_cast<uint32_t>(a.warps_g));
        const uint32_t wc1 = min(static_cast<uint32_t>(c * kDecWarps + kDecWarps), static_cast<uint32_t>(a.warps_g));
        const uint32_t cu0 = split_begin(U_g, a.warps_g, wc0), cu1 = split_begin(U_g, a.warps_g, wc1);
        const int cta_item0 = static_cast<int>(cu0 / npan_g);
        const int cta_items = cu1 > cu0 ? static_cast<int>((cu1 - 1) / npan_g) - cta_item0 + 1 : 0;
        float* cred = reinterpret_cast<float*>(dsm + a.off_p);
        for (int i = tid; i < cta_items * kDecWarps * 32; i += kDecThreads) cred[i] = 0.0f;
        if (tid < kMaxK) {   // every slot holds a valid expert even if the logits were not finite
            s_sel[tid] = 0;
            s_val[tid] = 0.0f;
        }
        __syncthreads();
        if constexpr (kSupplied) {
            // the caller's selection, pair j in slot j; an index outside [0, E) is clamped and
            // recorded as device error 1, as in the other paths
            if (tid < k) {
                int e = a.idx_in[tid];
                if (e < 0 || e >= E) {
                    if (c == 0) set_error(a.ws.err, kDevErrBadExpert);
                    e = min(max(e, 0), E - 1);
                }
                s_sel[tid] = e;
            }
        } else if constexpr (!wide) {
            // slot = number of experts that beat e, counted by tpe adjacent lanes per expert,
            // lane p over the float4 groups p, p + tpe, ... (a warp's loads are contiguous, free
            // of bank conflicts; E * tpe <= 512, E a multiple of 4)
            const int lg_tpe = E <= 64 ? 3 : (E <= 128 ? 2 : 1);
            const int tpe = 1 << lg_tpe;
            const int e = tid >> lg_tpe, part = tid & (tpe - 1);
            const bool live = e < E;
            const int nq = live ? E / 4 : 0;
            const float v = live ? slog[e] : 0.0f;
            const float4* row = reinterpret_cast<const float4*>(slog);
            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
            for (int q = part; q < nq; q += tpe) {
                const float4 o = row[q];
                r0 += beats(o.x, 4 * q, v, e);
                r1 += beats(o.y, 4 * q + 1, v, e);
                r2 += beats(o.z, 4 * q + 2, v, e);
                r3 += beats(o.w, 4 * q + 3, v, e);
            }
            int r = r0 + r1 + r2 + r3;
            for (int m = 1; m < tpe; m <<= 1) r += __shfl_xor_sync(0xffffffffu, r, m);
            if (live && part == 0 && r < k) {
                s_sel[r] = e;
                s_val[r] = v;
            }
        } else {
            if (router) rank_own_experts(slog, s_cnt, E, k, epc, c, a.sel, a.selv);
            grid_barrier(a.bar, ++nbar * G, a.ws.err, wait_ns);
            if (tid < k) {   // (clamped: after a given-up barrier the word may be stale)
                s_sel[tid] = min(max(__ldcg(a.sel + tid), 0), E - 1);
                s_val[tid] = __ldcg(a.selv + tid);
            }
        }
        __syncthreads();
        if (warp == 0 && lane < k) {   // sorted slot of pair j: selected experts with a lower index
            const int ej = s_sel[lane];
            int r = 0;
            if constexpr (kSupplied) {   // an expert the caller repeats takes one slot per pair, in pair order
                for (int i = 0; i < k; ++i) r += s_sel[i] < ej || (s_sel[i] == ej && i < lane);
            } else {
                for (int i = 0; i < k; ++i) r += s_sel[i] < ej;
            }
            s_e[r] = ej;
            s_pos[lane] = r;
        }
        __syncthreads();
        // The combine weights and the routing record need only the selection: they are worked
        // out once the CTA's first gate.up requests are in flight (s_w is next read in the
        // combine, several CTA barriers later).
        auto finish_routing = [&]() {
            if (warp == 0 && lane < k) {   // softmax over the k selected logits (slot 0's subtracted, sum in slot order)
                const int j = lane, ej = s_sel[j], r = s_pos[j];
                float wj;
                if constexpr (kSupplied) {
                    wj = a.w_in[j];
                } else {
                    const float m0 = s_val[0];
                    float sum = 0.0f;
                    for (int i = 0; i < k; ++i) sum += expf(s_val[i] - m0);
                    wj = expf(s_val[j] - m0) / sum;
                }
                s_w[j] = wj;
                if (c == 0 && a.idx_out) {
                    a.idx_out[l * k + j] = ej;
                    a.w_out[l * k + j] = wj;
                }
                if (c == 0) {
                    a.ws.idx[j] = ej;
                    a.ws.w[j] = wj;
                    a.ws.perm[r] = j;
                    a.ws.pos[j] = r;
                    a.ws.act_e[r] = ej;
                    a.ws.slot_info[r] = make_int4(ej, r, 1, 0);
                }
            }
            if (c == 0) {
                for (int e = tid; e <= E; e += kDecThreads) {
                    int n = 0;
                    for (int i = 0; i < k; ++i) n += s_sel[i] < e;
                    a.ws.offsets[e] = n;
                }
                if (tid == 0) *a.ws.n_active = k;
            }
        };

        // ---------------------------------------------------------------- G: gate.up partial sums
        const uint64_t pol = l2_evict_first_policy();
        if (tid == 0 && P.pf_bytes > 0) {   // this CTA's share of the caller's L2 hint
            const int64_t share = ((P.pf_bytes + G - 1) / G + 127) / 128 * 128;
            const int64_t off = static_cast<int64_t>(c) * share;
            if (off < P.pf_bytes) prefetch_l2(P.pf + off, static_cast<uint32_t>(min(share, P.pf_bytes - off)));
        }
        // The routed experts' down matrices, asked of L2 while gate.up streams (a hint): CTA c
        // takes a contiguous 1/G of the k matrices' bytes, in a few large bulk requests (each
        // bulk request costs the copy engine about the same whatever its size).
        auto prefetch_down = [&]() {
            if (tid != 0 || !a.prefetch_down) return;
            const int64_t total = static_cast<int64_t>(k) * a.dn_bytes;
            const int64_t share = ((total + G - 1) / G + 15) / 16 * 16;
            int64_t off = static_cast<int64_t>(c) * share;
            const int64_t end = min(total, off + share);
            while (off < end) {
                const int s = static_cast<int>(off / a.dn_bytes);
                const int64_t within = off - static_cast<int64_t>(s) * a.dn_bytes;
                const int64_t n = min(end - off, a.dn_bytes - within);
                prefetch_l2(P.w_dn + static_cast<int64_t>(s_e[s]) * a.dn_bytes + within, static_cast<uint32_t>(n));
                off += n;
            }
        };
        // Q8_0 down: the issue pointer as (slot, row tile, panel), advanced by increments:
        // slot-major, so that a CTA's units read the activations of one or two slots only.  The
        // first stages are requested as soon as the warp's gate.up units are done (they do not
        // depend on h), so they are in flight across the barrier.
        const uint32_t dring_addr = smem_addr(ring + warp * kStages * kSlotBytes);
        int dss = rd.item0 / nrt, dsrt = rd.item0 % nrt, dsb = rd.b0;
        const uint8_t* dsw = P.w_dn + static_cast<int64_t>(s_e[dss < k ? dss : 0]) * a.dn_bytes;
        auto issue_d = [&](int st) {
            issue_panel_block<FMT>(dring_addr + st * kSlotBytes, dsw, d, dsrt * 32, dsrt * 32 + 16, dsb, pol, 0);
            if (++dsb == npan_d) {
                dsb = 0;
                if (++dsrt == nrt) {
                    dsrt = 0;
                    if (++dss < k) dsw = P.w_dn + static_cast<int64_t>(s_e[dss]) * a.dn_bytes;
                }
            }
        };
        {
            const int n = rg.n;   // 0 for a warp past the split (more warps than units)
            unsigned char* wring = ring + warp * kStages * kSlotBytes;
            const uint32_t ring_addr = smem_addr(wring);
            // the issue pointer as (slot, tile, panel), advanced by increments
            int iss_s = rg.item0 / nt_g, iss_t = rg.item0 % nt_g, iss_b = rg.b0;
            const uint8_t* iss_w = P.w_gu + static_cast<int64_t>(s_e[iss_s < k ? iss_s : 0]) * a.gu_bytes;
            auto issue = [&](int st) {
                // SwiGLU: gate rows t*16.. and up rows f + t*16..; ReLU^2: rows t*32.. and t*32 + 16..
                const int rA = iss_t * (kSwiglu ? 16 : 32), rB = kSwiglu ? f + iss_t * 16 : iss_t * 32 + 16;
                issue_panel_block<FMT>(ring_addr + st * kSlotBytes, iss_w, kSwiglu ? 2 * f : f, rA, rB, iss_b, pol, 0);
                if (++iss_b == npan_g) {
                    iss_b = 0;
                    if (++iss_t == nt_g) {
                        iss_t = 0;
                        if (++iss_s < k) iss_w = P.w_gu + static_cast<int64_t>(s_e[iss_s]) * a.gu_bytes;
                    }
                }
            };
#pragma unroll
            for (int st = 0; st < kStages; ++st) {
                if (st < n) issue(st);
                cp_async_commit();
            }
            prefetch_down();   // after this warp's first gate.up requests
            finish_routing();   // while they are in flight
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            int cur_item = rg.item0, cur_b = rg.b0;
            for (int i0 = 0; i0 < n; i0 += kStages) {
#pragma unroll 1   // rolled: the kernel's code stays small (no faster unrolled on GB300)
                for (int st = 0; st < kStages; ++st) {
                    const int i = i0 + st;
                    if (i < n) {
                        cp_async_wait<kStages - 1>();
                        __syncwarp();
                        panel_mma<FMT>(wring + st * kSlotBytes, xh, d, cur_b, 1, 0, acc, split_l, d);
                        __syncwarp();   // every lane is done with the slot before it is refilled
                        if (i + kStages < n) issue(st);
                        cp_async_commit();
                        if (++cur_b == npan_g || i == n - 1) {
                            // this warp's share of the item, token column 0: lanes t == 0 hold rows
                            // g and g + 8 of blocks A and B (gate and up, or the tile's two halves)
                            if ((lane & 3) == 0) {
                                float* rr = cred + ((cur_item - cta_item0) * kDecWarps + warp) * 32;
                                const int g = lane >> 2;
                                rr[g] = acc[0][0];
                                rr[g + 8] = acc[0][2];
                                rr[16 + g] = acc[1][0];
                                rr[24 + g] = acc[1][2];
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[0][q] = acc[1][q] = 0.0f;
                            cur_b = 0;
                            ++cur_item;
                        }
                    }
                }
            }
            cp_async_wait<0>();
            if constexpr (kQ8) {
#pragma unroll
                for (int st = 0; st < kStages; ++st) {
                    if (st < rd.n) issue_d(st);
                    cp_async_commit();
                }
            }
        }
        // The CTA's record of each item it touched: its warps' partials in warp order (a warp
        // that did not touch the item adds zero), at the CTA's contributor slot of the item.
        __syncthreads();
        for (int i = tid; i < cta_items * 32; i += kDecThreads) {
            const int it = i >> 5, j = i & 31;
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) v += cred[(it * kDecWarps + w) * 32 + j];
            const uint32_t item = static_cast<uint32_t>(cta_item0 + it);
            const int cidx = c - static_cast<int>(split_owner(U_g, a.warps_g, item * npan_g) / kDecWarps);
            a.grec[(static_cast<int64_t>(item) * a.cov_g + cidx) * 32 + j] = v;
        }
        grid_barrier(a.bar, ++nbar * G, a.ws.err, wait_ns);

        if constexpr (kQ8) {
            // ---------------------------------------------------------------- D ring, then H
            // The down panel blocks do not depend on h: this warp's first ones are requested before
            // the activations are reduced.
            const int kf = k * f;
            __half* hs = reinterpret_cast<__half*>(xf);   // [k][f] hi, then [k][f] lo
            unsigned char* dring = ring + warp * kStages * kSlotBytes;
            // H: h = SiLU(gate) * up.  Each CTA sums the records (in contributor order) of the slots
            // its down units read, into its own f16 hi + lo copy of h, and writes them as fp32 too
            // (every slot is read by some CTA; CTAs that share a slot write the same values).
            int h_lo_q = 0, h_hi_q = 0;   // neurons [h_lo_q, h_hi_q) of the flattened [k][f]
            {
                const uint32_t w0 = min(static_cast<uint32_t>(c * kDecWarps), static_cast<uint32_t>(a.warps_d));
                const uint32_t w1 = min(static_cast<uint32_t>(c * kDecWarps + kDecWarps), static_cast<uint32_t>(a.warps_d));
                const uint32_t v0 = split_begin(U_d, a.warps_d, w0), v1 = split_begin(U_d, a.warps_d, w1);
                const uint32_t per_slot = static_cast<uint32_t>(nrt * npan_d);
                if (v1 > v0) {
                    h_lo_q = static_cast<int>(v0 / per_slot) * f;
                    h_hi_q = (static_cast<int>((v1 - 1) / per_slot) + 1) * f;
                }
            }
            int* gcov = reinterpret_cast<int*>(slog);     // CTAs that recorded each gate.up item (items_g <= 1024)
            for (int i = tid; i < static_cast<int>(items_g); i += kDecThreads) {
                const uint32_t u0 = static_cast<uint32_t>(i) * npan_g, u1 = u0 + npan_g - 1;
                gcov[i] = static_cast<int>(split_owner(U_g, a.warps_g, u1) / kDecWarps -
                                           split_owner(U_g, a.warps_g, u0) / kDecWarps) + 1;
            }
            __syncthreads();
            constexpr int kHB = 4;   // neurons per thread per batch: their first two records load together
            for (int q0 = h_lo_q + tid; q0 < h_hi_q; q0 += kHB * kDecThreads) {   // neuron q = item * 16 + j
                float g0[kHB], g1[kHB], u0[kHB], u1[kHB];
#pragma unroll
                for (int u = 0; u < kHB; ++u) {
                    const int q = q0 + u * kDecThreads;
                    g0[u] = g1[u] = u0[u] = u1[u] = 0.0f;
                    if (q < h_hi_q) {
                        const float* rec = a.grec + static_cast<int64_t>(q >> 4) * a.cov_g * 32 + (q & 15);
                        g0[u] = __ldcg(rec);
                        u0[u] = __ldcg(rec + 16);
                        if (gcov[q >> 4] > 1) {
                            g1[u] = __ldcg(rec + 32);
                            u1[u] = __ldcg(rec + 48);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kHB; ++u) {
                    const int q = q0 + u * kDecThreads;
                    if (q < h_hi_q) {
                        float zg = g0[u] + g1[u], zu = u0[u] + u1[u];   // records in contributor order
                        const float* rec = a.grec + static_cast<int64_t>(q >> 4) * a.cov_g * 32 + (q & 15);
                        for (int cc = 2; cc < gcov[q >> 4]; ++cc) {
                            zg += __ldcg(rec + cc * 32);
                            zu += __ldcg(rec + cc * 32 + 16);
                        }
                        float h = silu(zg) * zu;
                        if constexpr (AQ) {   // the down projection's input through the coder (a warp: one block of 32)
                            const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h))));
                            h = q8_0_coded_value(h, amax);
                        }
                        const __half hi = __float2half_rn(h);
                        hs[q] = hi;
                        hs[kf + q] = __float2half_rn(h - __half2float(hi));
                        a.ws.h[q] = h;
                    }
                }
            }
            __syncthreads();

            // ---------------------------------------------------------------- D: down partial sums
            // A unit is one 32-neuron panel of a 32-row tile of one slot's down matrix (two 16-row
            // MMA blocks, the gate.up panel product with h as the activations).
            if (rd.n > 0) {
                const int n = rd.n;
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                int cur_item = rd.item0, cur_s = rd.item0 / nrt, cur_rt = rd.item0 % nrt, cur_b = rd.b0, cur_c = rd.c0;
                for (int i0 = 0; i0 < n; i0 += kStages) {
#pragma unroll 1   // rolled: the kernel's code stays small (no faster unrolled on GB300)
                    for (int st = 0; st < kStages; ++st) {
                        const int i = i0 + st;
                        if (i < n) {
                            cp_async_wait<kStages - 1>();
                            __syncwarp();
                            panel_mma<FMT>(dring + st * kSlotBytes, hs + cur_s * f, f, cur_b, 1, 0, acc, true, kf);
                            __syncwarp();   // every lane is done with the slot before it is refilled
                            if (i + kStages < n) issue_d(st);
                            cp_async_commit();
                            if (++cur_b == npan_d || i == n - 1) {
                                if ((lane & 3) == 0) {   // rows g, g + 8 of both blocks, token column 0
                                    float* rec = a.drec + (static_cast<int64_t>(cur_item) * a.cov_d + cur_c) * 32;
                                    const int g = lane >> 2;
                                    rec[g] = acc[0][0];
                                    rec[g + 8] = acc[0][2];
                                    rec[16 + g] = acc[1][0];
                                    rec[24 + g] = acc[1][2];
                                }
#pragma unroll
                                for (int q = 0; q < 4; ++q) acc[0][q] = acc[1][q] = 0.0f;
                                cur_b = 0;
                                cur_c = 0;
                                ++cur_item;
                                if (++cur_rt == nrt) {
                                    cur_rt = 0;
                                    ++cur_s;
                                }
                            }
                        }
                    }
                }
            }
            cp_async_wait<0>();
            grid_barrier(a.bar, ++nbar * G, a.ws.err, wait_ns);
            if (l + 1 < a.n_layers) request_router(a.lp[l + 1].W);   // the ring is free until the next gate.up

            // ---------------------------------------------------------------- C: combine
            // Row tile rt (32 outputs) is combined by CTA rt mod G: y of each slot (its records in
            // contributor order), then out[r] = sum over the pairs j in order of w_j * y_{slot(j)}[r].
            float* s_y = slog;   // [k][32] (kMaxK * 32 == kMaxE floats)
            static_assert(kMaxK * 32 <= kMaxE, "combine buffer");
            for (int rt = c; rt < nrt; rt += G) {
                for (int task = tid; task < k * 32; task += kDecThreads) {
                    const int s = task >> 5, r = task & 31;
                    const uint32_t item = static_cast<uint32_t>(s * nrt + rt);
                    const int nc = item_contributors(U_d, a.warps_d, npan_d, item);
                    const float* rec = a.drec + static_cast<int64_t>(item) * a.cov_d * 32 + r;
                    float v[8];   // the first 8 records in one batch (one L2 round trip)
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = q < nc ? __ldcg(rec + q * 32) : 0.0f;
                    float y = v[0];   // records in contributor order
#pragma unroll
                    for (int q = 1; q < 8; ++q) y += v[q];
                    for (int cc = 8; cc < nc; ++cc) y += __ldcg(rec + cc * 32);
                    s_y[s * 32 + r] = y;
                }
                __syncthreads();
                if (tid < 32) {
                    float o = 0.0f;
                    for (int j = 0; j < k; ++j) o = fmaf(s_w[j], s_y[s_pos[j] * 32 + tid], o);
                    a.out[static_cast<int64_t>(l) * d + rt * 32 + tid] = o;
                }
                __syncthreads();
            }
        } else {
            // ------------------------------------------------------------ H (NVFP4)
            // h = max(z * ts, 0)^2 (ReLU^2, 32-neuron items) or SiLU(zg * ts) * (zu * ts) (SwiGLU,
            // items of 16 gate + 16 up rows) for the slots this CTA's down units read (fp32, in
            // region B), the records of each item summed in contributor order; then which
            // 16-neuron groups hold a non-zero h (the only ones the down projection reads).
            float* hf = xf;                                   // [cta slots][f]
            int* gact = reinterpret_cast<int*>(slog);         // [cta slots][f/16] active flags
            float* dred = reinterpret_cast<float*>(ring);     // [cta items][16 warps][256] down partials
            const uint32_t dw0 = min(static_cast<uint32_t>(c * kDecWarps), static_cast<uint32_t>(a.warps_d));
            const uint32_t dw1 = min(static_cast<uint32_t>(c * kDecWarps + kDecWarps), static_cast<uint32_t>(a.warps_d));
            const uint32_t dv0 = split_begin(U_d, a.warps_d, dw0), dv1 = split_begin(U_d, a.warps_d, dw1);
            const uint32_t per_slot = static_cast<uint32_t>(nrt * npan_d);
            const int h_s0 = static_cast<int>(dv0 / per_slot);
            const int h_ns = dv1 > dv0 ? static_cast<int>((dv1 - 1) / per_slot) - h_s0 + 1 : 0;
            const int d_item0 = static_cast<int>(dv0 / npan_d);
            const int d_items = dv1 > dv0 ? static_cast<int>((dv1 - 1) / npan_d) - d_item0 + 1 : 0;
            for (int i = tid; i < d_items * kDecWarps * 256; i += kDecThreads) dred[i] = 0.0f;
            constexpr int kHB = kSwiglu ? 4 : 8;   // neurons per thread per batch: their first two records load together
            constexpr int kLg = kSwiglu ? 4 : 5;   // log2 of the neurons per gate.up item
            // the record word of neuron qq within its item (SwiGLU: the gate row; the up row is 16 later)
            auto rec_of = [&](int qq) {
                return a.grec + static_cast<int64_t>(qq >> kLg) * a.cov_g * 32 + (qq & ((1 << kLg) - 1));
            };
            const int hn = h_ns * f;
            for (int q0 = tid; q0 < hn; q0 += kHB * kDecThreads) {
                float v0[kHB], v1[kHB], w0[kHB], w1[kHB];   // (gate or z) and up, first two records
                int ncs[kHB];
#pragma unroll
                for (int u = 0; u < kHB; ++u) {
                    const int q = q0 + u * kDecThreads;
                    v0[u] = v1[u] = w0[u] = w1[u] = 0.0f;
                    ncs[u] = 0;
                    if (q < hn) {
                        const int qq = h_s0 * f + q;          // neuron of the flattened [k][f]
                        const uint32_t item = static_cast<uint32_t>(qq >> kLg);
                        ncs[u] = static_cast<int>(split_owner(U_g, a.warps_g, (item + 1) * npan_g - 1) / kDecWarps -
                                                  split_owner(U_g, a.warps_g, item * npan_g) / kDecWarps) + 1;
                        const float* rec = rec_of(qq);
                        v0[u] = __ldcg(rec);
                        if (kSwiglu) w0[u] = __ldcg(rec + 16);
                        if (ncs[u] > 1) {
                            v1[u] = __ldcg(rec + 32);
                            if (kSwiglu) w1[u] = __ldcg(rec + 48);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kHB; ++u) {
                    const int q = q0 + u * kDecThreads;
                    if (q < hn) {
                        const int qq = h_s0 * f + q;
                        const float* rec = rec_of(qq);
                        float z = v0[u] + v1[u], zu = w0[u] + w1[u];   // records in contributor order
                        for (int cc = 2; cc < ncs[u]; ++cc) {
                            z += __ldcg(rec + cc * 32);
                            if (kSwiglu) zu += __ldcg(rec + cc * 32 + 16);
                        }
                        const float ts = P.gu_ts[s_e[qq / f]];
                        float h;
                        if constexpr (kSwiglu) {
                            h = silu(z * ts) * (zu * ts);
                        } else {
                            z *= ts;
                            h = z > 0.0f ? z * z : 0.0f;
                        }
                        hf[q] = h;
                        a.ws.h[qq] = h;
                    }
                }
            }
            __syncthreads();
            for (int gi = tid; gi < h_ns * (f / 16); gi += kDecThreads) {
                bool any = false;
#pragma unroll
                for (int j = 0; j < 16; ++j) any |= hf[gi * 16 + j] != 0.0f;
                gact[gi] = any ? 1 : 0;
            }
            __syncthreads();

            // ------------------------------------------------------------ D (NVFP4)
            // Units (slot, 256-row tile, group of 16 neurons), group fastest.  Lane l owns rows
            // 8l .. 8l+7 of the tile: per active group 16 code words (one per neuron) and 8 row
            // scales; the products are exact in fp32 (e2m1 x f32 h), summed over the group's
            // neurons in order, then scaled by each row's E4M3 scale.  Inactive groups are not
            // read.  Two active groups' loads are in flight per warp.
            if (rd.n > 0) {
                const int64_t grp_bytes = 16 * (d / 2) + d;     // one group record of a matrix
                int scan_item = rd.item0, scan_g = rd.b0, left = rd.n;
                int acc_item = -1;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                auto flush = [&]() {
                    if (acc_item >= 0) {
                        float* rr = dred + ((acc_item - d_item0) * kDecWarps + warp) * 256 + lane * 8;
                        *reinterpret_cast<float4*>(rr) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                        *reinterpret_cast<float4*>(rr + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
                };
                // the next active unit of the range (-1: none left)
                auto next_active = [&](int& g_out) -> int {
                    while (left > 0) {
                        const int it = scan_item, g = scan_g;
                        --left;
                        if (++scan_g == npan_d) {
                            scan_g = 0;
                            ++scan_item;
                        }
                        if (gact[(it / nrt - h_s0) * npan_d + g]) {
                            g_out = g;
                            return it;
                        }
                    }
                    return -1;
                };
                auto load = [&](int it, int g, uint32_t (&cw)[16], uint2& sc) {
                    const int sl = it / nrt, rt = it % nrt;
                    const uint8_t* base = P.w_dn + static_cast<int64_t>(s_e[sl]) * a.dn_bytes + g * grp_bytes;
#pragma unroll
                    for (int j = 0; j < 16; ++j) cw[j] = ldg_stream4(base + j * (d / 2) + rt * 128 + lane * 4);
                    sc = ldg_stream8(base + 16 * (d / 2) + rt * 256 + lane * 8);
                };
                auto compute = [&](int it, int g, const uint32_t (&cw)[16], const uint2& sc) {
                    if (it != acc_item) {
                        flush();
                        acc_item = it;
                    }
                    const float* hv = hf + (it / nrt - h_s0) * f + 16 * g;
                    uint64_t part[4] = {0, 0, 0, 0};   // rows (2by, 2by+1): one packed fmaf pair per code byte
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float h = hv[j];
                        const uint64_t hh = pack_f32x2(h, h);
#pragma unroll
                        for (int by = 0; by < 4; ++by) {
                            const float2 v = e2m1x2_to_f32x2((cw[j] >> (8 * by)) & 0xffu);   // rows 2by, 2by+1
                            fma_f32x2(part[by], pack_f32x2(v.x, v.y), hh);
                        }
                    }
#pragma unroll
                    for (int by = 0; by < 4; ++by) {
                        const float2 pv = unpack_f32x2(part[by]);
                        const uint32_t sw = by < 2 ? sc.x : sc.y;
                        const int r = 2 * by;
                        acc[r] = fmaf(e4m3_to_f32((sw >> (8 * (r & 3))) & 0xffu), pv.x, acc[r]);
                        acc[r + 1] = fmaf(e4m3_to_f32((sw >> (8 * ((r + 1) & 3))) & 0xffu), pv.y, acc[r + 1]);
                    }
                };
                uint32_t cw0[16], cw1[16];
                uint2 sc0, sc1;
                int g0 = 0, g1 = 0;
                int it0 = next_active(g0);
                if (it0 >= 0) load(it0, g0, cw0, sc0);
                while (it0 >= 0) {
                    const int it1 = next_active(g1);
                    if (it1 >= 0) load(it1, g1, cw1, sc1);
                    compute(it0, g0, cw0, sc0);
                    if (it1 < 0) break;
                    it0 = next_active(g0);
                    if (it0 >= 0) load(it0, g0, cw0, sc0);
                    compute(it1, g1, cw1, sc1);
                }
                flush();
            }
            // The CTA's record of each down item it touched: its warps' partials in warp order.
            __syncthreads();
            for (int i = tid; i < d_items * 256; i += kDecThreads) {
                const int it = i >> 8, r = i & 255;
                float v = 0.0f;
#pragma unroll 4
                for (int w = 0; w < kDecWarps; ++w) v += dred[(it * kDecWarps + w) * 256 + r];
                const uint32_t item = static_cast<uint32_t>(d_item0 + it);
                const int cidx = c - static_cast<int>(split_owner(U_d, a.warps_d, item * npan_d) / kDecWarps);
                a.drec[(static_cast<int64_t>(item) * a.cov_d + cidx) * 256 + r] = v;
            }
            grid_barrier(a.bar, ++nbar * G, a.ws.err, wait_ns);
            if (l + 1 < a.n_layers) request_router(a.lp[l + 1].W);   // the ring is free until the next gate.up

            // ------------------------------------------------------------ C (NVFP4)
            // 32-row chunk q of the output is combined by CTA q mod G: y of each slot (its CTA
            // records in order, times the down tensor scale), then the pairs in order j.
            float* s_y = slog;   // [k][32]
            for (int q = c; q < d / 32; q += G) {
                const int rt = q / 8, off = (q % 8) * 32;
                for (int task = tid; task < k * 32; task += kDecThreads) {
                    const int sl = task >> 5, r = task & 31;
                    const uint32_t item = static_cast<uint32_t>(sl * nrt + rt);
                    const int nc = static_cast<int>(split_owner(U_d, a.warps_d, (item + 1) * npan_d - 1) / kDecWarps -
                                                    split_owner(U_d, a.warps_d, item * npan_d) / kDecWarps) + 1;
                    const float* rec = a.drec + static_cast<int64_t>(item) * a.cov_d * 256 + off + r;
                    float v[4];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) v[cc] = cc < nc ? __ldcg(rec + cc * 256) : 0.0f;
                    float y = ((v[0] + v[1]) + v[2]) + v[3];   // records in contributor order
                    for (int cc = 4; cc < nc; ++cc) y += __ldcg(rec + cc * 256);
                    s_y[sl * 32 + r] = y * P.dn_ts[s_e[sl]];
                }
                __syncthreads();
                if (tid < 32) {
                    float o = 0.0f;
                    for (int j = 0; j < k; ++j) o = fmaf(s_w[j], s_y[s_pos[j] * 32 + tid], o);
                    a.out[static_cast<int64_t>(l) * d + q * 32 + tid] = o;
                }
                __syncthreads();
            }
        }
        // ---------------------------------------------------------------- N: the next layer's input
        // x_{l+1} = bf16(out_l / sqrt(mean(out_l^2) + eps)), the sum of squares in the order of the
        // stand-alone RMS-norm kernel (threads t < 256 take elements t, t + 256, ...; warp sums;
        // the 8 warp sums in order), so a stack equals its layers glued by that kernel bitwise.
        if (l + 1 < a.n_layers || a.x_next) {
            grid_barrier(a.bar, ++nbar * G, a.ws.err, wait_ns);
            const float* ol = a.out + static_cast<int64_t>(l) * d;
            float* wsum = slog;
            // out_l into shared memory, loaded in batches of 8 per thread (one L2 round trip per
            // batch instead of one per element)
            for (int base = 0; base < d; base += 8 * kDecThreads) {
                float v[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int i = base + m * kDecThreads + tid;
                    v[m] = i < d ? __ldcg(ol + i) : 0.0f;
                }
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int i = base + m * kDecThreads + tid;
                    if (i < d) xf[i] = v[m];
                }
            }
            __syncthreads();
            if (tid < 256) {
                float ss = 0.0f;
                for (int i = tid; i < d; i += 256) ss = fmaf(xf[i], xf[i], ss);
                ss = warp_sum(ss);
                if (lane == 0) wsum[warp] = ss;
            }
            __syncthreads();
            float tot = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) tot += wsum[i];
            const float inv = rsqrtf(tot / static_cast<float>(d) + a.eps);
            for (int i = tid; i < d; i += kDecThreads) {   // (whole warps: d is a multiple of 256)
                const __nv_bfloat16 xb = __float2bfloat16_rn(xf[i] * inv);
                const float xv = __bfloat162float(xb);
                xf[i] = xv;
                if constexpr (AQ) {   // the experts' x through the coder (a warp: one block of 32), hi + lo
                    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(xv))));
                    const float cv = q8_0_coded_value(xv, amax);
                    const __half hi = __float2half_rn(cv);
                    xh[i] = hi;
                    xh[d + i] = __float2half_rn(cv - __half2float(hi));
                } else {
                    xh[i] = __float2half_rn(xv);
                }
                if (c == 0 && a.x_next) a.x_next[static_cast<int64_t>(l) * d + i] = __bfloat16_as_ushort(xb);
            }
            __syncthreads();   // (slog is read again by the next layer's selection)
        }
    }
    // The last CTA to finish resets the barrier counters for the next call: every CTA has
    // passed (or given up on) all of its barriers by now.
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(a.bar + 1, 1) == G - 1) {
            a.bar[0] = 0;
            a.bar[1] = 0;
        }
    }
}

// ------------------------------------------------------------------------------ host side
// Dynamic shared memory the kernel is configured for (with its static arrays, within the
// 227 KB one CTA may hold).
size_t decode_max_smem() { return 220 * 1024; }

namespace {
bool g_decode_ok[64] = {};
int g_decode_ctas[64] = {};

template <int FMT, int ACT, int ROUTE, bool AQ = false>
bool configure_one() {
    const int max_smem = static_cast<int>(decode_max_smem());
    if (cudaFuncSetAttribute(decode_layer_kernel<FMT, ACT, ROUTE, AQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             max_smem) != cudaSuccess)
        return false;
    int per_sm = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel<FMT, ACT, ROUTE, AQ>,
                                                                        kDecThreads, max_smem);
    return e == cudaSuccess && per_sm >= 1;
}
}  // namespace

// Dynamic shared memory limit, cooperative-launch support and one-CTA-per-SM residency
// (once per device, with that device current).
cudaError_t configure_decode_kernel(int dev, int num_sms) {
    g_decode_ok[dev] = false;
    int coop = 0;
    cudaError_t e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) return e;
    if (!coop) return cudaSuccess;
    if (!configure_one<MOE_W_Q8_0, MOE_ACT_SWIGLU, kRouteLocal>() ||
        !configure_one<MOE_W_Q8_0, MOE_ACT_SWIGLU, kRouteWide>() ||
        !configure_one<MOE_W_Q8_0, MOE_ACT_SWIGLU, kRouteSupplied>() ||
        !configure_one<MOE_W_Q8_0, MOE_ACT_SWIGLU, kRouteLocal, true>() ||
        !configure_one<MOE_W_Q8_0, MOE_ACT_SWIGLU, kRouteWide, true>() ||
        !configure_one<MOE_W_Q8_0, MOE_ACT_SWIGLU, kRouteSupplied, true>() ||
        !configure_one<MOE_W_INT8PC, MOE_ACT_SWIGLU, kRouteLocal>() ||
        !configure_one<MOE_W_INT8PC, MOE_ACT_SWIGLU, kRouteWide>() ||
        !configure_one<MOE_W_INT8PC, MOE_ACT_SWIGLU, kRouteSupplied>() ||
        !configure_one<MOE_W_NVFP4, MOE_ACT_RELU2, kRouteLocal>() ||
        !configure_one<MOE_W_NVFP4, MOE_ACT_RELU2, kRouteWide>() ||
        !configure_one<MOE_W_NVFP4, MOE_ACT_RELU2, kRouteSupplied>() ||
        !configure_one<MOE_W_NVFP4, MOE_ACT_SWIGLU, kRouteLocal>() ||
        !configure_one<MOE_W_NVFP4, MOE_ACT_SWIGLU, kRouteWide>() ||
        !configure_one<MOE_W_NVFP4, MOE_ACT_SWIGLU, kRouteSupplied>()) {
        (void)cudaGetLastError();
        return cudaSuccess;   // the separate kernels serve every shape
    }
    g_decode_ok[dev] = true;
    g_decode_ctas[dev] = num_sms < kMaxDecodeCtas ? num_sms : kMaxDecodeCtas;
    return cudaSuccess;
}

// CTAs of the decode kernel on this device (0: not available).
int decode_ctas(int dev) { return (dev >= 0 && dev < 64 && g_decode_ok[dev]) ? g_decode_ctas[dev] : 0; }

template <int FMT, int ACT, bool AQ = false>
static cudaError_t launch_decode_route(const cudaLaunchConfig_t& cfg, const DecodeArgs& a, int route) {
    if (route == kRouteSupplied) return cudaLaunchKernelEx(&cfg, decode_layer_kernel<FMT, ACT, kRouteSupplied, AQ>, a);
    if (route == kRouteWide) return cudaLaunchKernelEx(&cfg, decode_layer_kernel<FMT, ACT, kRouteWide, AQ>, a);
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel<FMT, ACT, kRouteLocal, AQ>, a);
}

cudaError_t launch_decode_layer(const DecodeArgs& a, int wfmt, int act, size_t smem, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const int route = a.idx_in ? kRouteSupplied : (a.E > kLocalRankMaxE ? kRouteWide : kRouteLocal);
    if (wfmt == MOE_W_Q8_0 && a.act_q) return launch_decode_route<MOE_W_Q8_0, MOE_ACT_SWIGLU, true>(cfg, a, route);
    if (wfmt == MOE_W_Q8_0) return launch_decode_route<MOE_W_Q8_0, MOE_ACT_SWIGLU>(cfg, a, route);
    if (wfmt == MOE_W_INT8PC) return launch_decode_route<MOE_W_INT8PC, MOE_ACT_SWIGLU>(cfg, a, route);
    if (act == MOE_ACT_SWIGLU) return launch_decode_route<MOE_W_NVFP4, MOE_ACT_SWIGLU>(cfg, a, route);
    return launch_decode_route<MOE_W_NVFP4, MOE_ACT_RELU2>(cfg, a, route);
}

}  // namespace moe
