// api.cu -- the C ABI of libmoe (include/moe.h): host-side validation, workspace layout
// and the launch sequence of one MoE layer.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace moe {

// launchers (pack.cu, route.cu, gemv.cu)
cudaError_t launch_q8_0_quantize(const float*, int64_t, int64_t, int64_t, int, void*, cudaStream_t);
cudaError_t launch_nvfp4_pack(const float*, int64_t, int64_t, int64_t, int, void*, float*, cudaStream_t);
cudaError_t launch_act_q8_0(const void*, int, int64_t, int64_t, float*, uint16_t*, uint16_t*, int, cudaStream_t);
cudaError_t launch_int8pc_quantize(const float*, int64_t, int64_t, int64_t, int, void*, cudaStream_t);
cudaError_t launch_router_logits(const void*, int, const float*, int64_t, int64_t, int64_t, float*, cudaStream_t);
cudaError_t launch_topk_softmax(const float*, int64_t, int64_t, int, int32_t*, float*, cudaStream_t);
cudaError_t launch_route_small(const float*, const int32_t*, const float*, int64_t, int64_t, int, int,
                               const Workspace&, cudaStream_t);
cudaError_t launch_permute_large(const int32_t*, const float*, int64_t, int64_t, int, int, const Workspace&,
                                 cudaStream_t);
cudaError_t launch_route_decode(const void*, int, const float*, int64_t, int64_t, int64_t, int, int, const Workspace&,
                                cudaStream_t);
bool route_decode_fits(int64_t, int64_t, int64_t);
cudaError_t configure_gemv_kernels();
cudaError_t launch_gate_up_gemv(const ExpertArgs&, int, int, int, cudaStream_t);
cudaError_t launch_down_gemv(const ExpertArgs&, int, int, cudaStream_t);
size_t down_nv_mma_smem(int, int);
cudaError_t launch_down_q8_t1(const ExpertArgs&, cudaStream_t);
cudaError_t launch_combine(const float*, const int32_t*, const float*, int64_t, int, int64_t, float*, cudaStream_t);
cudaError_t launch_rmsnorm_bf16(const float*, int64_t, int64_t, float, uint16_t*, cudaStream_t);
cudaError_t configure_gemm_kernels();
cudaError_t configure_route_kernels();
cudaError_t launch_expert_gemm(const ExpertArgs&, int, int, int, int, int, int, cudaStream_t);
cudaError_t launch_gather_x_f16(const ExpertArgs&, int, cudaStream_t);
cudaError_t configure_decode_kernel(int, int);
int decode_ctas(int);
size_t decode_smem_plan(int, int, int, int, int, int, int, int*, int*);
size_t decode_ring_bytes();
size_t decode_max_smem();
cudaError_t launch_decode_layer(const DecodeArgs&, int, int, size_t, int, cudaStream_t);


namespace {

constexpr int64_t kMaxDim = 1 << 16;
constexpr int64_t kMaxTokens = 1 << 20;
constexpr int64_t kMaxF = 32768;     // group-mask words per slot fit the kernels' 64-word array
constexpr int kSmallT = 32;          // route_small handles up to 32 tokens
constexpr int kSmallPairs = 1024;    // ... and up to 1024 pairs
constexpr int64_t kFusedRouteLogits = 4096;   // ... and up to 4096 logits (the routing CTA keeps them on chip)
constexpr size_t kSmemBudget = 96 * 1024;        // token rows staged per expert CTA (plus the 55 KB ring)
constexpr int64_t kPrefetchBudget = 64ll << 20;   // down weights prefetched into L2 (of 126 MB)
constexpr size_t kNvMmaSmem = 112 * 1024;         // NVFP4 tensor-core down: stage ring + h planes + group lists (2 CTAs per SM)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes of one quantised matrix [rows, cols] in the format (every layout of a format has them).
int64_t matrix_bytes(int wfmt, int64_t rows, int64_t cols) {
    if (wfmt == MOE_W_Q8_0) return static_cast<int64_t>(moe_q8_0_bytes(rows, cols));
    if (wfmt == MOE_W_NVFP4) return static_cast<int64_t>(moe_nvfp4_bytes(rows, cols));
    return static_cast<int64_t>(moe_int8pc_bytes(rows, cols));
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-device one-time kernel attribute setup (dynamic shared memory above 48 KB) and the
// device's SM count.
int g_num_sms[64] = {};

cudaError_t ensure_configured(int* num_sms) {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = configure_gemv_kernels();
        if (e == cudaSuccess) e = configure_gemm_kernels();
        if (e == cudaSuccess) e = configure_route_kernels();
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = configure_decode_kernel(dev, g_num_sms[dev]);
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    *num_sms = g_num_sms[dev];
    return cudaSuccess;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct Plan {
    int64_t T, P;
    int slot_cap;       // min(E, P)
    int nchunk;
    int gwords;
    int tt_gu, tt_dn;
    bool small_route;   // T <= 32 and P <= 1024: routing and permutation in one CTA
    bool fuse_combine;  // the down kernel's last CTA per row tile combines (one item per thread)
    bool prefetch_down; // gate.up CTAs prefetch the routed experts' down weights into L2
    bool gemm;          // expert GEMMs on the tensor cores instead of the GEMVs
    bool down_t1;       // one token, Q8_0 SwiGLU, k in {1,2,4,8}: the row-tile down kernel combines
    int nv_split;       // NVFP4 down with fused combine: group splits per (row tile, slot)
    bool nv_mma;        // NVFP4 down on the tensor cores (tt_dn tokens per pass)
    bool decode1;       // one token, Q8_0 SwiGLU: the shape fits the one-kernel decode layer
};

// Router experts per routing CTA of the one-kernel decode layer (0: E too large for `ctas`).
int decode_epc(int64_t E, int ctas) {
    for (int epc : {1, 2, 4, 8})
        if (E % epc == 0 && E / epc <= ctas) return epc;
    return 0;
}

// The one-kernel decode layer splits U_g = k * f/16 * d/32 gate.up panel units and
// U_d = d/32 * k * f/32 down units evenly over the warps of `ctas` CTAs (16 each).
struct DecodeSplit {
    int64_t U_g, U_d, warps_g, warps_d;
    int64_t npan_g, npan_d;  // panels per gate.up item, units per down item
    int64_t cov_g;       // CTAs whose ranges can touch one gate.up item (records per item)
    int64_t cov_d;       // Q8_0: warps, NVFP4: CTAs whose ranges can touch one down item
    int64_t cta_items;   // gate.up items one CTA's range can touch
    int64_t cta_items_d; // NVFP4: down items one CTA's range can touch
    int64_t cta_slots;   // NVFP4: slots whose activations one CTA's down units read
    int64_t items_d;     // down items
    int64_t rec_d;       // floats per down record (32 rows, or 256 rows for NVFP4)
};

// The most items of npan units that one CTA's range (16 warps of an even split of U over W)
// touches.
int64_t cta_max_items(int64_t U, int64_t W, int64_t npan) {
    int64_t m = 0;
    for (int64_t c = 0; 16 * c < W; ++c) {
        const int64_t w0 = 16 * c, w1 = std::min(16 * c + 16, W);
        const int64_t u0 = w0 * U / W, u1 = w1 * U / W;
        if (u1 > u0) m = std::max(m, (u1 - 1) / npan - u0 / npan + 1);
    }
    return m;
}

// Q8_0 SwiGLU: gate.up units (slot, 16-neuron tile, 32-column panel), down units (slot,
// 32-row tile, 32-neuron panel).  NVFP4: gate.up units (slot, 32-neuron tile (ReLU^2) or
// 16-neuron tile of gate and up rows (SwiGLU), 64-column panel), down units (slot, 256-row
// tile, 16-neuron group).
DecodeSplit decode_split(const moe_layer_desc* d, int64_t ctas) {
    DecodeSplit sp{};
    const bool q8 = d->wfmt != MOE_W_NVFP4;   // 32-column int8 panels (Q8_0, per-channel int8)
    sp.npan_g = q8 ? d->d / 32 : d->d / 64;
    sp.npan_d = q8 ? d->f / 32 : d->f / 16;
    const int64_t items_g = static_cast<int64_t>(d->k) * (d->act == MOE_ACT_SWIGLU ? d->f / 16 : d->f / 32);
    sp.items_d = static_cast<int64_t>(d->k) * (q8 ? d->d / 32 : d->d / 256);
    sp.rec_d = q8 ? 32 : 256;
    sp.U_g = items_g * sp.npan_g;
    sp.U_d = sp.items_d * sp.npan_d;
    sp.warps_g = std::min<int64_t>(16 * ctas, sp.U_g);
    sp.warps_d = std::min<int64_t>(16 * ctas, sp.U_d);
    // a range of at least Lmin units meets at most ceil(npan / Lmin) + 1 items; +2 for margin
    const int64_t lcta = std::max<int64_t>(1, sp.U_g / ((sp.warps_g + 15) / 16));   // units per CTA, at least
    sp.cov_g = (sp.npan_g + lcta - 1) / lcta + 2;
    const int64_t lwd = std::max<int64_t>(1, q8 ? sp.U_d / sp.warps_d : sp.U_d / ((sp.warps_d + 15) / 16));
    sp.cov_d = (sp.npan_d + lwd - 1) / lwd + 2;
    sp.cta_items = cta_max_items(sp.U_g, sp.warps_g, sp.npan_g);
    sp.cta_items_d = q8 ? 0 : cta_max_items(sp.U_d, sp.warps_d, sp.npan_d);
    sp.cta_slots = q8 ? 0 : cta_max_items(sp.U_d, sp.warps_d, sp.npan_d * (d->d / 256));
    return sp;
}

// The one-kernel decode layer's shape limits (any device): one token, Q8_0 or per-channel int8
// SwiGLU, or NVFP4 (ReLU^2 or SwiGLU), the router-weight slice of a routing CTA and x within its shared memory, and 32-bit
// unit arithmetic.
// The input type the one-kernel layer's shared-memory plan takes: coded activations (Q8_0
// values need about 19 significant bits) travel as two f16 planes, like an fp32 input.
int decode_xt(const moe_layer_desc* d, int xt) { return d->act_quant == MOE_ACTQ_Q8_0 ? MOE_F32 : xt; }

bool decode_shape_ok(const moe_layer_desc* d, int64_t T, int xt) {
    if (T != 1 || d->path != MOE_PATH_AUTO) return false;
    const bool q8 = (d->wfmt == MOE_W_Q8_0 || d->wfmt == MOE_W_INT8PC) && d->act == MOE_ACT_SWIGLU;
    const bool nv = d->wfmt == MOE_W_NVFP4;   // ReLU^2 (latent experts) or SwiGLU
    if (!q8 && !nv) return false;
    if (d->d > 8192 || d->f % 32 != 0) return false;
    if (q8 && d->k * d->f > 16384) return false;   // h of every slot in shared memory
    if (decode_smem_plan(d->wfmt, static_cast<int>(d->d), static_cast<int>(d->f), d->k, xt, 1, 1, nullptr, nullptr) >
        decode_max_smem())
        return false;
    const int epc = decode_epc(d->E, kMaxDecodeCtas);
    if (epc == 0 || static_cast<size_t>(d->d * epc * 4 + epc * 1024) > decode_ring_bytes()) return false;
    const DecodeSplit sp = decode_split(d, kMaxDecodeCtas);   // the most warps: the largest products
    return (sp.U_g + 1) * sp.warps_g < (int64_t(1) << 32) && (sp.U_d + 1) * sp.warps_d < (int64_t(1) << 32);
}

// With `ctas` CTAs on this device: the kernel's shared memory, including the per-warp
// gate.up partials of one CTA's items, within what the kernel is configured for.
bool decode_split_fits(const moe_layer_desc* d, const DecodeSplit& sp, int xt) {
    if (decode_smem_plan(d->wfmt, static_cast<int>(d->d), static_cast<int>(d->f), d->k, xt,
                         static_cast<int>(sp.cta_items), static_cast<int>(sp.cta_slots), nullptr,
                         nullptr) > decode_max_smem())
        return false;
    if (d->wfmt == MOE_W_NVFP4) {
        // the down partials of the CTA's items fit the ring; its slots' group flags fit 1024 words
        if (static_cast<size_t>(sp.cta_items_d) * 16 * 256 * sizeof(float) > decode_ring_bytes()) return false;
        if (sp.cta_slots * (d->f / 16) > 1024) return false;
    } else if (static_cast<int64_t>(d->k) * (d->f / 16) > 1024) {
        return false;   // contributor counts of the gate.up items fit 1024 words
    }
    return true;
}

// The GEMM path tiles rows by 128 (SwiGLU gate.up: 64 neurons' gate and up rows) and K by 64.
bool gemm_shape_ok(const moe_layer_desc* d) {
    if (d->wfmt == MOE_W_INT8PC) return false;   // per-channel int8 runs on the GEMV kernels
    if (d->flags & MOE_FLAG_HOST_WEIGHTS) return false;   // TMA loads device memory only
    if (d->f % 64 != 0 || d->d % 64 != 0) return false;
    if (d->act == MOE_ACT_RELU2 && d->f % 128 != 0) return false;
    return true;
}

Plan make_plan(const moe_layer_desc* d, int64_t T, int xt = MOE_BF16) {
    Plan p{};
    p.T = T;
    p.P = T * d->k;
    p.slot_cap = static_cast<int>(std::min<int64_t>(d->E, p.P));
    p.nchunk = static_cast<int>((p.P + 1023) / 1024);
    p.gwords = static_cast<int>((d->f / 16 + 31) / 32);
    // Token tiles: the staged activations take shared memory per CTA, and with it CTAs per SM,
    // so tiles are sized for twice the average pairs per routed expert (room for a skewed
    // routing); an expert with more tokens loops over further tiles.
    const int64_t slots = std::max<int64_t>(1, std::min<int64_t>(d->E, p.P));
    const int64_t want = 2 * ((p.P + slots - 1) / slots);
    const int64_t tmax = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(8, T), want));
    // staged activations: f16 (bf16 inputs) or f16 hi + lo (fp32 inputs; h always) per element
    const int64_t x_bytes = (xt == MOE_F32) ? 4 : 2;
    p.tt_gu = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tmax, kSmemBudget / (x_bytes * d->d))));
    // NVFP4 down: token tiles of at most 2 (two CTAs per SM fit in registers; a 4-token tile
    // leaves one per SM, and a few tokens per expert is the common case)
    const int64_t dn_cap = (d->wfmt == MOE_W_NVFP4) ? 2 : 8;
    p.tt_dn = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(std::min(tmax, dn_cap), kSmemBudget / (4 * d->f))));
    // the tile counts are powers of two up to 8 (the kernels specialise 1, 2, 4, 8)
    auto pow2 = [](int v) { return v >= 8 ? 8 : (v >= 4 ? 4 : (v >= 2 ? 2 : 1)); };   // (rounds down)
    p.tt_gu = pow2(p.tt_gu);
    p.tt_dn = pow2(p.tt_dn);
    p.small_route = (T <= kSmallT && p.P <= kSmallPairs && T * d->E <= kFusedRouteLogits) &&
                    route_decode_fits(T, d->d, d->E);
    const int64_t rows_per_tile = (d->wfmt == MOE_W_NVFP4) ? 256 : 32;
    p.fuse_combine = T * rows_per_tile <= 256;
    const int64_t dn_bytes = matrix_bytes(d->wfmt, d->d, d->f);
    p.prefetch_down = static_cast<int64_t>(p.slot_cap) * dn_bytes <= kPrefetchBudget &&
                      !(d->flags & MOE_FLAG_HOST_DOWN);   // no bulk L2 prefetch of host memory
    // many tokens per expert (at least 8 on average): tensor-core GEMMs
    p.gemm = gemm_shape_ok(d) && (d->path == MOE_PATH_GEMM || (d->path == MOE_PATH_AUTO && p.P >= 8 * d->E));
    if (p.gemm) p.fuse_combine = false;
    p.down_t1 = !p.gemm && T == 1 && d->wfmt == MOE_W_Q8_0 && d->act == MOE_ACT_SWIGLU &&
                (d->k == 1 || d->k == 2 || d->k == 4 || d->k == 8) && d->f / 32 >= 8 / d->k && d->d % 16 == 0;
    if (p.down_t1) p.fuse_combine = true;   // the down kernel writes the output rows
    p.nv_split = (!p.gemm && d->wfmt == MOE_W_NVFP4 && p.fuse_combine && T == 1 && (d->f / 16) >= 4 * 8) ? 4 : 1;
    // NVFP4 down at two or more tokens: tensor cores, tokens in passes of 8, 16 or 32 (as many
    // as T asks for and the f16 h planes leave room for in shared memory)
    p.nv_mma = !p.gemm && d->wfmt == MOE_W_NVFP4 && !p.fuse_combine && T >= 2 &&
               down_nv_mma_smem(8, static_cast<int>(d->f)) <= kNvMmaSmem;
    if (p.nv_mma) {
        int tt = 8;
        while (tt < 32 && tt < T && down_nv_mma_smem(2 * tt, static_cast<int>(d->f)) <= kNvMmaSmem) tt *= 2;
        p.tt_dn = tt;
    }
    // (coded activations: Q8_0 SwiGLU, with x carried as two f16 planes like an fp32 input)
    p.decode1 = !p.gemm &&
                (d->act_quant == MOE_ACTQ_NONE || (d->wfmt == MOE_W_Q8_0 && d->act == MOE_ACT_SWIGLU)) &&
                decode_shape_ok(d, T, decode_xt(d, xt));
    return p;
}

struct Layout {
    size_t err, route_ctr, n_active, wait_limit, row_ctr, logits, rpart, idx, w, offsets, perm, pos, act_e, slot_info, chunk_cnt,
        local_rank, gmask, h, y, xs_hi, xs_lo, h_hi, h_lo, dec_bar, dec_sel, dec_grec, dec_drec, xnext, xq, total;
};

// The control region at the start of every workspace: a 256-byte header (the error word,
// the routing counter, the one-kernel layer's barrier counters, the test-only wait limit)
// and the fused combine's row-tile counters, sized for the largest d.  Neither offset nor
// size depends on the layer's shape or T, so one workspace (or the no-allocation scratch)
// serves layers of any shape and calls of any token count in any order.
constexpr size_t kCtrlHeaderBytes = 256;
constexpr size_t kRowCtrBytes = sizeof(int32_t) * (kMaxDim / 32);   // 8 KiB
constexpr size_t kCtrlBytes = kCtrlHeaderBytes + kRowCtrBytes;

// Workspace regions for T tokens (each 256-byte aligned).  The control words (err,
// route_ctr, the one-kernel layer's two barrier counters, row_ctr) come first, at offsets
// that depend neither on T nor on the layer's shape: they must be zero before a call and
// are left zero, so one workspace serves calls of any token count and any layer shape in
// any order.
Layout layout_for(const moe_layer_desc* d, int64_t T) {
    const Plan p = make_plan(d, T);
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    L.err = 0;
    L.route_ctr = 4;
    L.n_active = 8;
    L.dec_bar = 16;   // [2]: grid-barrier arrivals, CTAs finished (one-kernel layer)
    L.wait_limit = 32;   // int64: grid-barrier wait limit in ns, 0 = the default second
    L.row_ctr = kCtrlHeaderBytes;
    off = kCtrlBytes;
    L.logits = take(sizeof(float) * T * d->E);
    L.rpart = take(p.small_route ? sizeof(float) * T * d->E * 32 : 0);
    L.idx = take(sizeof(int32_t) * p.P);
    L.w = take(sizeof(float) * p.P);
    L.offsets = take(sizeof(int32_t) * (d->E + 1));
    L.perm = take(sizeof(int32_t) * p.P);
    L.pos = take(sizeof(int32_t) * p.P);
    L.act_e = take(sizeof(int32_t) * p.slot_cap);
    L.slot_info = take(sizeof(int4) * p.slot_cap);
    L.chunk_cnt = take(sizeof(int32_t) * p.nchunk * d->E);
    L.local_rank = take(sizeof(int32_t) * p.P);
    L.gmask = take(sizeof(uint32_t) * p.slot_cap * p.gwords);
    L.h = take(sizeof(float) * p.P * d->f);
    L.y = take(sizeof(float) * p.P * d->d * p.nv_split);   // NVFP4 split partials
    // f16 planes of the tensor-core path (the lo plane of x is used by fp32 inputs only)
    const size_t xs = p.gemm ? sizeof(uint16_t) * p.P * d->d : 0;
    const size_t hs = p.gemm ? sizeof(uint16_t) * p.P * d->f : 0;
    L.xs_hi = take(xs);
    L.xs_lo = take(xs);
    L.h_hi = take(hs);
    L.h_lo = take(hs);
    // the one-kernel decode layer's counters (zero between calls) and partial sums
    const bool dec = p.decode1;
    // (sized for the most CTAs any device can give the kernel: more CTAs, more records per item)
    const DecodeSplit sp = decode_split(d, kMaxDecodeCtas);
    L.dec_sel = take(dec ? sizeof(int32_t) * 2 * kMaxK : 0);
    L.dec_grec = take(dec ? sizeof(float) * 32 * (sp.U_g / sp.npan_g) * sp.cov_g : 0);
    L.dec_drec = take(dec ? sizeof(float) * sp.rec_d * sp.items_d * sp.cov_d : 0);
    L.xnext = take(T == 1 ? sizeof(uint16_t) * d->d : 0);   // a stack's next input (one token)
    L.xq = take(d->act_quant ? sizeof(float) * T * d->d : 0);   // the coded expert input (MOE_ACTQ_Q8_0)
    L.total = off;
    return L;
}

}  // namespace

size_t workspace_control_bytes() { return kCtrlBytes; }

namespace {

Workspace bind(void* base, const Layout& L) {
    char* b = static_cast<char*>(base);
    Workspace w{};
    w.err = reinterpret_cast<int32_t*>(b + L.err);
    w.route_ctr = reinterpret_cast<int32_t*>(b + L.route_ctr);
    w.row_ctr = reinterpret_cast<int32_t*>(b + L.row_ctr);
    w.n_active = reinterpret_cast<int32_t*>(b + L.n_active);
    w.logits = reinterpret_cast<float*>(b + L.logits);
    w.rpart = reinterpret_cast<float*>(b + L.rpart);
    w.idx = reinterpret_cast<int32_t*>(b + L.idx);
    w.w = reinterpret_cast<float*>(b + L.w);
    w.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
    w.perm = reinterpret_cast<int32_t*>(b + L.perm);
    w.pos = reinterpret_cast<int32_t*>(b + L.pos);
    w.act_e = reinterpret_cast<int32_t*>(b + L.act_e);
    w.slot_info = reinterpret_cast<int4*>(b + L.slot_info);
    w.chunk_cnt = reinterpret_cast<int32_t*>(b + L.chunk_cnt);
    w.local_rank = reinterpret_cast<int32_t*>(b + L.local_rank);
    w.gmask = reinterpret_cast<uint32_t*>(b + L.gmask);
    w.h = reinterpret_cast<float*>(b + L.h);
    w.y = reinterpret_cast<float*>(b + L.y);
    w.xs_hi = reinterpret_cast<uint16_t*>(b + L.xs_hi);
    w.xs_lo = reinterpret_cast<uint16_t*>(b + L.xs_lo);
    w.h_hi = reinterpret_cast<uint16_t*>(b + L.h_hi);
    w.h_lo = reinterpret_cast<uint16_t*>(b + L.h_lo);
    return w;
}

moe_status validate_desc(const moe_layer_desc* d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->act != MOE_ACT_SWIGLU && d->act != MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
    if (d->wfmt != MOE_W_Q8_0 && d->wfmt != MOE_W_NVFP4 && d->wfmt != MOE_W_INT8PC) return MOE_ERR_INVALID_ARG;
    if (d->path != MOE_PATH_AUTO && d->path != MOE_PATH_GEMV && d->path != MOE_PATH_GEMM) return MOE_ERR_INVALID_ARG;
    if (d->E < 1 || d->E > kMaxE || d->E % 4 != 0) return MOE_ERR_SHAPE;
    if (d->k < 1 || d->k > kMaxK || d->k > d->E) return MOE_ERR_INVALID_ARG;
    if (d->d < 256 || d->d > kMaxDim || d->d % 256 != 0) return MOE_ERR_SHAPE;
    const int64_t fq = (d->wfmt == MOE_W_NVFP4) ? 64 : 32;
    if (d->f < fq || d->f > kMaxF || d->f % fq != 0) return MOE_ERR_SHAPE;
    if (d->act == MOE_ACT_RELU2 && d->f % 32 != 0) return MOE_ERR_SHAPE;
    if (!d->router_w || !d->w_gate_up || !d->w_down) return MOE_ERR_INVALID_ARG;
    if (d->wfmt == MOE_W_NVFP4 && (!d->gate_up_tscale || !d->down_tscale)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(d->router_w) || !aligned16(d->w_gate_up) || !aligned16(d->w_down)) return MOE_ERR_ALIGNMENT;
    if (d->l2_prefetch && (d->l2_prefetch_bytes < 0 || !aligned16(d->l2_prefetch))) return MOE_ERR_ALIGNMENT;
    if (d->act_quant != MOE_ACTQ_NONE && d->act_quant != MOE_ACTQ_Q8_0) return MOE_ERR_INVALID_ARG;
    if (d->act_quant == MOE_ACTQ_Q8_0 && d->wfmt != MOE_W_Q8_0) return MOE_ERR_UNSUPPORTED;
    if (d->flags & ~MOE_FLAG_HOST_WEIGHTS) return MOE_ERR_INVALID_ARG;   // unknown bits
    if ((d->flags & MOE_FLAG_HOST_WEIGHTS) && d->path == MOE_PATH_GEMM) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Every expert stack a MOE_FLAG_HOST_* bit names is a host allocation (page-locked, mapped) that
// the device reads at the same pointer.
bool host_weights_ok(const moe_layer_desc* d) {
    for (int bit : {MOE_FLAG_HOST_GATE_UP, MOE_FLAG_HOST_DOWN}) {
        if (!(d->flags & bit)) continue;
        const void* p = bit == MOE_FLAG_HOST_GATE_UP ? d->w_gate_up : d->w_down;
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        if (at.type != cudaMemoryTypeHost || at.devicePointer != p) return false;
    }
    return true;
}

// The one-kernel decode arguments for n layers of descs[0]'s shape (pointers per layer), on
// the current device; false when the device or the shape cannot run it.
bool fill_decode_args(const moe_layer_desc* descs, int n, const void* x, int xt, void* workspace, const Layout& L,
                      const Workspace& ws, DecodeArgs* a, int* ctas_out, size_t* smem_out) {
    const moe_layer_desc* desc = descs;
    const Plan p = make_plan(desc, 1, xt);
    if (!p.decode1 || n < 1 || n > kMaxStackLayers) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const int ctas = decode_ctas(dev);
    const int epc = decode_epc(desc->E, ctas);
    const DecodeSplit sp = decode_split(desc, std::max(1, ctas));
    const int xt_planes = decode_xt(desc, xt);   // the shared-memory plan's input type: fp32 = two f16 planes
    if (ctas <= 0 || epc <= 0 || !decode_split_fits(desc, sp, xt_planes)) return false;
    for (int l = 1; l < n; ++l)   // one kernel serves the stack only if every layer codes (or not) and reads alike
        if (descs[l].act_quant != desc->act_quant || descs[l].flags != desc->flags) return false;
    char* base = static_cast<char*>(workspace);
    *a = DecodeArgs{};
    a->x = x;
    a->xt = xt;
    a->act_q = desc->act_quant == MOE_ACTQ_Q8_0 ? 1 : 0;
    a->d = static_cast<int>(desc->d);
    a->f = static_cast<int>(desc->f);
    a->E = static_cast<int>(desc->E);
    a->k = desc->k;
    a->epc = epc;
    // the routed experts' whole down matrices into L2 (Q8_0 and SwiGLU: every byte is read;
    // NVFP4 ReLU^2 reads only the active groups, so a whole-matrix prefetch would fetch bytes
    // that are skipped)
    a->prefetch_down = (p.prefetch_down && (desc->wfmt == MOE_W_Q8_0 || desc->act == MOE_ACT_SWIGLU)) ? 1 : 0;
    // warps that share each phase's panel range: all of them, or one per unit
    a->warps_g = static_cast<int>(sp.warps_g);
    a->warps_d = static_cast<int>(sp.warps_d);
    a->cov_g = static_cast<int>(sp.cov_g);
    a->cov_d = static_cast<int>(sp.cov_d);
    a->cta_items = static_cast<int>(sp.cta_items);
    a->cta_items_d = static_cast<int>(sp.cta_items_d);
    const int64_t rows_gu = desc->act == MOE_ACT_SWIGLU ? 2 * desc->f : desc->f;
    a->gu_bytes = matrix_bytes(desc->wfmt, rows_gu, desc->d);
    a->dn_bytes = matrix_bytes(desc->wfmt, desc->d, desc->f);
    *smem_out = decode_smem_plan(desc->wfmt, a->d, a->f, a->k, xt_planes, a->cta_items, static_cast<int>(sp.cta_slots),
                                 &a->off_c, &a->off_p);
    a->n_layers = n;
    for (int l = 0; l < n; ++l) {
        a->lp[l].W = descs[l].router_w;
        a->lp[l].w_gu = static_cast<const uint8_t*>(descs[l].w_gate_up);
        a->lp[l].w_dn = static_cast<const uint8_t*>(descs[l].w_down);
        a->lp[l].pf = static_cast<const uint8_t*>(descs[l].l2_prefetch);
        a->lp[l].pf_bytes = descs[l].l2_prefetch ? (descs[l].l2_prefetch_bytes & ~static_cast<int64_t>(15)) : 0;
        a->lp[l].gu_ts = descs[l].gate_up_tscale;
        a->lp[l].dn_ts = descs[l].down_tscale;
    }
    a->ws = ws;
    a->bar = reinterpret_cast<int32_t*>(base + L.dec_bar);
    a->sel = reinterpret_cast<int32_t*>(base + L.dec_sel);
    a->selv = reinterpret_cast<float*>(base + L.dec_sel + sizeof(int32_t) * kMaxK);
    a->grec = reinterpret_cast<float*>(base + L.dec_grec);
    a->drec = reinterpret_cast<float*>(base + L.dec_drec);
    *ctas_out = ctas;
    return true;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return 10300; }

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: a pointer is NULL or an argument is out of range";
        case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE: a dimension is not a supported multiple or is too large";
        case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT: a pointer is not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: this combination is not built";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime call failed";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: a kernel recorded an error";
    }
    return "unknown moe_status";
}

size_t moe_q8_0_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0 || cols % 32 != 0) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols / 32) * 34;
}

size_t moe_int8pc_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0 || cols % 32 != 0) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols) + 4 * static_cast<size_t>(rows);
}

size_t moe_nvfp4_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0 || cols % 16 != 0) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols) / 2 + static_cast<size_t>(rows) * cols / 16;
}

moe_status moe_quantize_q8_0(const float* src, int64_t n_mat, int64_t rows, int64_t cols, moe_layout layout,
                             void* dst, moe_stream_t stream) {
    if (!src || !dst || n_mat < 0) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_LAYOUT_CANONICAL && layout != MOE_LAYOUT_DEVICE) return MOE_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 32 != 0 || rows > kMaxTokens || cols > kMaxDim)
        return MOE_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_ALIGNMENT;
    if (n_mat == 0) return MOE_OK;
    return cuda_status(launch_q8_0_quantize(src, n_mat, rows, cols, layout, dst, stream));
}

moe_status moe_quantize_int8pc(const float* src, int64_t n_mat, int64_t rows, int64_t cols, moe_layout layout,
                               void* dst, moe_stream_t stream) {
    if (!src || !dst || n_mat < 0) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_LAYOUT_CANONICAL && layout != MOE_LAYOUT_DEVICE) return MOE_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 32 != 0 || rows > kMaxTokens || cols > kMaxDim)
        return MOE_ERR_SHAPE;
    if (n_mat > 65535) return MOE_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_ALIGNMENT;
    if (n_mat == 0) return MOE_OK;
    return cuda_status(launch_int8pc_quantize(src, n_mat, rows, cols, layout, dst, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_pack_nvfp4(const float* src, int64_t n_mat, int64_t rows, int64_t cols, moe_layout layout, void* dst,
                          float* tensor_scale, moe_stream_t stream) {
    if (!src || !dst || !tensor_scale || n_mat < 0) return MOE_ERR_INVALID_ARG;
    if (layout != MOE_LAYOUT_CANONICAL && layout != MOE_LAYOUT_DEVICE && layout != MOE_LAYOUT_NEURON)
        return MOE_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || rows % 32 != 0 || cols % 64 != 0 || rows > kMaxTokens || cols > kMaxDim)
        return MOE_ERR_SHAPE;
    if (n_mat > 65535) return MOE_ERR_SHAPE;
    if (!aligned16(src) || !aligned16(dst) || (reinterpret_cast<uintptr_t>(tensor_scale) & 3u)) return MOE_ERR_ALIGNMENT;
    if (n_mat == 0) return MOE_OK;
    return cuda_status(launch_nvfp4_pack(src, n_mat, rows, cols, layout, dst, tensor_scale, stream));
}

moe_status moe_quantize_act_q8_0(const void* x, moe_dtype xt, int64_t rows, int64_t cols, float* out,
                                 moe_stream_t stream) {
    if (!x || !out) return MOE_ERR_INVALID_ARG;
    if (xt != MOE_F32 && xt != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (rows < 0 || cols <= 0 || cols % 32 != 0 || rows > kMaxTokens * kMaxK || cols > kMaxF * 2) return MOE_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
    if (rows == 0) return MOE_OK;
    int num_sms = 0;
    if (ensure_configured(&num_sms) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_act_q8_0(x, xt, rows, cols, out, nullptr, nullptr, num_sms,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_router_workspace_bytes(int64_t T, int64_t E) {
    if (T < 0 || E < 1) return 0;
    return round_up(sizeof(float) * static_cast<size_t>(T) * static_cast<size_t>(E), 256);
}

moe_status moe_router_topk(const void* x, moe_dtype xt, const float* W, int64_t T, int64_t d, int64_t E, int k,
                           int32_t* idx, float* w, float* logits, void* workspace, size_t ws_bytes,
                           moe_stream_t stream) {
    if (!x || !W || !idx || !w) return MOE_ERR_INVALID_ARG;
    if (xt != MOE_F32 && xt != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (T < 0 || T > kMaxTokens) return MOE_ERR_SHAPE;
    if (E < 4 || E > kMaxE || E % 4 != 0) return MOE_ERR_SHAPE;
    if (k < 1 || k > kMaxK || k > E) return MOE_ERR_INVALID_ARG;
    if (d < 256 || d > kMaxDim || d % 256 != 0) return MOE_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(W) || !aligned16(idx) || !aligned16(w) || (logits && !aligned16(logits)))
        return MOE_ERR_ALIGNMENT;
    float* lg = logits;
    if (!lg) {
        if (!workspace || ws_bytes < moe_router_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE;
        if (!aligned16(workspace)) return MOE_ERR_ALIGNMENT;
        lg = static_cast<float*>(workspace);
    }
    if (T == 0) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_router_logits(x, xt, W, T, d, E, lg, s);
    if (e == cudaSuccess) e = launch_topk_softmax(lg, T, E, k, idx, w, s);
    return cuda_status(e);
}

size_t moe_layer_workspace_bytes(const moe_layer_desc* desc, int64_t T_max) {
    if (validate_desc(desc) != MOE_OK || T_max < 1 || T_max > kMaxTokens) return 0;
    // Regions grow with T inside each routing regime; the fused small-batch routing also
    // needs a partial-sum buffer, so take the larger of the two regimes' layouts.
    int64_t t_small = std::min<int64_t>(T_max, kSmallT);
    t_small = std::min<int64_t>(t_small, kSmallPairs / desc->k);
    t_small = std::min<int64_t>(t_small, kFusedRouteLogits / desc->E);
    size_t n = layout_for(desc, T_max).total;
    if (t_small >= 1) n = std::max(n, layout_for(desc, t_small).total);
    n = std::max(n, layout_for(desc, 1).total);   // one token may take the one-kernel decode layer
    return n;
}

moe_status moe_layer_forward(const moe_layer_desc* desc, const void* x, moe_dtype xt, int64_t T,
                             const int32_t* idx_in, const float* w_in, float* out, void* workspace,
                             size_t ws_bytes, const moe_trace* trace, moe_stream_t stream) {
    moe_status st = validate_desc(desc);
    if (st != MOE_OK) return st;
    if (xt != MOE_F32 && xt != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (T < 0 || T > kMaxTokens) return MOE_ERR_SHAPE;
    if (T == 0) return MOE_OK;                 // an empty batch: its (possibly NULL) buffers are not touched
    if (!x || !out) return MOE_ERR_INVALID_ARG;
    if ((idx_in == nullptr) != (w_in == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
    if (idx_in && (!aligned16(idx_in) || !aligned16(w_in))) return MOE_ERR_ALIGNMENT;
    if (!workspace) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_ALIGNMENT;
    const Layout L = layout_for(desc, T);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (desc->path == MOE_PATH_GEMM && !gemm_shape_ok(desc)) return MOE_ERR_UNSUPPORTED;
    if (!host_weights_ok(desc)) return MOE_ERR_INVALID_ARG;

    int num_sms = 0;
    cudaError_t e = ensure_configured(&num_sms);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the experts read fp32 coded values on the activation-quantised path
    const bool actq = desc->act_quant == MOE_ACTQ_Q8_0;
    const int xt_exp = actq ? MOE_F32 : xt;
    const Plan p = make_plan(desc, T, xt_exp);
    const Workspace ws = bind(workspace, L);
    const int k = desc->k;

    auto mark = [&](int i) {
        if (trace && trace->stage_events[i] && e == cudaSuccess)
            e = cudaEventRecordWithFlags(static_cast<cudaEvent_t>(trace->stage_events[i]), s,
                                         cudaEventRecordExternal);   // a real record node under capture
    };
    // optional copies of the intermediates (device to device, on the stream)
    auto copy_trace = [&]() -> moe_status {
        if (!trace) return MOE_OK;
        auto cp = [&](void* dst, const void* src, size_t bytes) {
            if (dst && e == cudaSuccess) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s);
        };
        if (!idx_in) cp(trace->logits, ws.logits, sizeof(float) * T * desc->E);
        cp(trace->idx, ws.idx, sizeof(int32_t) * p.P);
        cp(trace->w, ws.w, sizeof(float) * p.P);
        cp(trace->offsets, ws.offsets, sizeof(int32_t) * (desc->E + 1));
        cp(trace->perm, ws.perm, sizeof(int32_t) * p.P);
        cp(trace->pos, ws.pos, sizeof(int32_t) * p.P);
        cp(trace->h, ws.h, sizeof(float) * p.P * desc->f);
        return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };

    mark(0);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    // One token: the whole layer as one cooperative kernel when the device and the shape allow
    // it (with supplied routing the kernel skips the router and the selection).
    if (p.decode1) {
        DecodeArgs a{};
        int ctas = 0;
        size_t smem = 0;
        if (fill_decode_args(desc, 1, x, xt, workspace, L, ws, &a, &ctas, &smem)) {
            a.out = out;
            a.idx_in = idx_in;
            a.w_in = w_in;
            e = launch_decode_layer(a, desc->wfmt, desc->act, smem, ctas, s);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
            for (int i = 1; i <= 4; ++i) mark(i);   // one kernel: the inner boundaries coincide
            if (e != cudaSuccess) return MOE_ERR_CUDA;
            return copy_trace();
        }
    }
    // 1. router + top-k + softmax, 2. permutation by expert
    if (p.small_route && !idx_in) {
        e = launch_route_decode(x, xt, desc->router_w, T, desc->d, desc->E, k, p.gwords, ws, s);
    } else if (p.small_route) {
        e = launch_route_small(nullptr, idx_in, w_in, T, desc->E, k, p.gwords, ws, s);
    } else {
        if (!idx_in) {
            e = launch_router_logits(x, xt, desc->router_w, T, desc->d, desc->E, ws.logits, s);
            if (e == cudaSuccess) e = launch_topk_softmax(ws.logits, T, desc->E, k, ws.idx, ws.w, s);
        }
        if (e == cudaSuccess) e = launch_permute_large(idx_in, w_in, T, desc->E, k, p.gwords, ws, s);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    // 3. gate.up + activation + group mask, 4. sparse down (+ combine), 5. combine
    ExpertArgs a{};
    a.x = x;
    a.xt = xt;
    if (actq) {   // the experts' input: x coded per block of 32 (Q8_0), as the values the codes stand for
        float* xq = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.xq);
        if ((e = launch_act_q8_0(x, xt, T, desc->d, xq, nullptr, nullptr, num_sms, s)) != cudaSuccess)
            return MOE_ERR_CUDA;
        a.x = xq;
        a.xt = MOE_F32;
    }
    a.d = static_cast<int>(desc->d);
    a.f = static_cast<int>(desc->f);
    a.k = k;
    a.rows_gu = static_cast<int>(desc->act == MOE_ACT_SWIGLU ? 2 * desc->f : desc->f);
    a.tt_gu = p.tt_gu;
    a.tt_dn = p.tt_dn;
    {   // warps per gate.up tile: at most 4, and each warp should stream at least 12 K panels
        // (fewer, longer panel runs per warp cost parallelism at d = 2816, and 8 warps of 24
        // panels were slower than 4 of 48 at d = 6144)
        const int npan = static_cast<int>(desc->wfmt == MOE_W_NVFP4 ? desc->d / 64 : desc->d / 32);
        int wpt = 4;
        while (wpt > 1 && npan / wpt < 12) wpt /= 2;
        a.gu_wpt = wpt;
    }
    a.gwords = p.gwords;
    a.T = static_cast<int>(T);
    a.P = static_cast<int>(p.P);
    a.fuse_combine = p.fuse_combine ? 1 : 0;
    a.prefetch_down = p.prefetch_down ? 1 : 0;
    a.nv_split = p.nv_split;
    a.nv_mma = p.nv_mma ? 1 : 0;
    a.out = out;
    a.w_gu = static_cast<const uint8_t*>(desc->w_gate_up);
    a.w_dn = static_cast<const uint8_t*>(desc->w_down);
    a.gu_bytes = matrix_bytes(desc->wfmt, a.rows_gu, desc->d);
    a.dn_bytes = matrix_bytes(desc->wfmt, desc->d, desc->f);
    a.pf = static_cast<const uint8_t*>(desc->l2_prefetch);
    a.pf_bytes = desc->l2_prefetch ? (desc->l2_prefetch_bytes & ~static_cast<int64_t>(15)) : 0;
    a.gu_ts = desc->gate_up_tscale;
    a.dn_ts = desc->down_tscale;
    a.ws = ws;
    mark(1);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (p.gemm) {
        e = launch_gather_x_f16(a, num_sms, s);
        if (e == cudaSuccess) e = launch_expert_gemm(a, 0, desc->wfmt, desc->act, p.slot_cap, static_cast<int>(desc->E), num_sms, s);
    } else {
        e = launch_gate_up_gemv(a, desc->wfmt, desc->act, p.slot_cap, s);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (actq) {   // h coded in place, and its f16 planes on the tensor-core path
        e = launch_act_q8_0(ws.h, MOE_F32, p.P, desc->f, ws.h, p.gemm ? ws.h_hi : nullptr, p.gemm ? ws.h_lo : nullptr,
                            num_sms, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(2);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (p.gemm) e = launch_expert_gemm(a, 1, desc->wfmt, desc->act, p.slot_cap, static_cast<int>(desc->E), num_sms, s);
    else if (p.down_t1 && !idx_in) e = launch_down_q8_t1(a, s);   // supplied routing may repeat an expert
    else e = launch_down_gemv(a, desc->wfmt, p.slot_cap, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    mark(3);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (!p.fuse_combine) {
        if ((e = launch_combine(ws.w, ws.pos, ws.y, T, k, desc->d, out, s)) != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(4);
    if (e != cudaSuccess) return MOE_ERR_CUDA;

    return copy_trace();
    return MOE_OK;
}

int32_t moe_layer_forward_launches(const moe_layer_desc* desc, int64_t T, int32_t routing_supplied) {
    if (validate_desc(desc) != MOE_OK || T < 0 || T > kMaxTokens) return -1;
    if (T == 0) return 0;
    const Plan p = make_plan(desc, T);
    if (p.decode1) {   // the one-kernel decode layer, when this device runs it
        int num_sms = 0, dev = 0;
        if (ensure_configured(&num_sms) == cudaSuccess && cudaGetDevice(&dev) == cudaSuccess &&
            decode_epc(desc->E, decode_ctas(dev)) > 0 &&
            decode_split_fits(desc, decode_split(desc, std::max(1, decode_ctas(dev))), decode_xt(desc, MOE_BF16)))
            return 1;
    }
    int n = 0;
    if (p.small_route) n += 1;                              // routing + permutation in one launch
    else n += (routing_supplied ? 0 : 2) + 3;               // router, top-k; rank, scan, scatter
    n += 2;                                                 // gate.up, down
    if (p.gemm) n += 1;                                     // sorted f16 copy of x
    if (!p.fuse_combine) n += 1;                            // combine
    if (desc->act_quant) n += 2;                            // the coded x and h
    return n;
}

// Layers of one shape (the first descriptor's d, f, E, k, activation and format).
static moe_status validate_stack(const moe_layer_desc* descs, int32_t n_layers) {
    if (!descs || n_layers < 1) return MOE_ERR_INVALID_ARG;
    for (int32_t l = 0; l < n_layers; ++l) {
        const moe_status st = validate_desc(descs + l);
        if (st != MOE_OK) return st;
        const moe_layer_desc& a = descs[0];
        const moe_layer_desc& b = descs[l];
        if (a.d != b.d || a.f != b.f || a.E != b.E || a.k != b.k || a.act != b.act || a.wfmt != b.wfmt ||
            a.path != b.path)
            return MOE_ERR_SHAPE;
    }
    return MOE_OK;
}

moe_status moe_stack_forward(const moe_layer_desc* descs, int32_t n_layers, const void* x, moe_dtype xt, float eps,
                             float* outs, uint16_t* x_next, int32_t* idx, float* w, void* workspace, size_t ws_bytes,
                             moe_stream_t stream) {
    moe_status st = validate_stack(descs, n_layers);
    if (st != MOE_OK) return st;
    if (xt != MOE_F32 && xt != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (!x || !outs || (idx == nullptr) != (w == nullptr) || !(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(outs) || (x_next && !aligned16(x_next))) return MOE_ERR_ALIGNMENT;
    if ((idx && (reinterpret_cast<uintptr_t>(idx) & 3u)) || (w && (reinterpret_cast<uintptr_t>(w) & 3u)))
        return MOE_ERR_ALIGNMENT;
    if (!workspace) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_ERR_ALIGNMENT;
    const Layout L = layout_for(descs, 1);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    for (int32_t l = 0; l < n_layers; ++l)
        if (!host_weights_ok(descs + l)) return MOE_ERR_INVALID_ARG;
    int num_sms = 0;
    if (ensure_configured(&num_sms) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t d = descs[0].d, k = descs[0].k;
    // the whole stack as one cooperative kernel
    {
        DecodeArgs a{};
        int ctas = 0;
        size_t smem = 0;
        if (fill_decode_args(descs, n_layers, x, xt, workspace, L, bind(workspace, L), &a, &ctas, &smem)) {
            a.out = outs;
            a.eps = eps;
            a.x_next = x_next;
            a.idx_out = idx;
            a.w_out = w;
            return cuda_status(launch_decode_layer(a, descs->wfmt, descs->act, smem, ctas, s));
        }
    }
    // otherwise layer by layer, the RMS-norm glue between them
    uint16_t* scratch = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + L.xnext);
    const void* xl = x;
    moe_dtype xtl = xt;
    for (int32_t l = 0; l < n_layers; ++l) {
        moe_trace tr{};
        tr.idx = idx ? idx + l * k : nullptr;
        tr.w = w ? w + l * k : nullptr;
        st = moe_layer_forward(descs + l, xl, xtl, 1, nullptr, nullptr, outs + l * d, workspace, ws_bytes,
                               idx ? &tr : nullptr, stream);
        if (st != MOE_OK) return st;
        const bool last = l + 1 == n_layers;
        if (last && !x_next) break;
        uint16_t* xn = x_next ? x_next + l * d : scratch;
        if (launch_rmsnorm_bf16(outs + l * d, 1, d, eps, xn, s) != cudaSuccess) return MOE_ERR_CUDA;
        xl = xn;
        xtl = MOE_BF16;
    }
    return MOE_OK;
}

int32_t moe_stack_forward_launches(const moe_layer_desc* descs, int32_t n_layers, int32_t with_x_next) {
    if (validate_stack(descs, n_layers) != MOE_OK) return -1;
    bool uniform = true;   // (the one-kernel stack needs every layer to code, and read its weights, alike)
    for (int32_t l = 1; l < n_layers; ++l)
        uniform = uniform && descs[l].act_quant == descs[0].act_quant && descs[l].flags == descs[0].flags;
    const int32_t one = moe_layer_forward_launches(descs, 1, 0);
    if (one == 1 && uniform && n_layers <= kMaxStackLayers) return 1;
    int32_t n = 0;   // layer by layer, the RMS-norm after each
    for (int32_t l = 0; l < n_layers; ++l) n += moe_layer_forward_launches(descs + l, 1, 0) + 1;
    return n - (with_x_next ? 0 : 1);
}

moe_status moe_rmsnorm_bf16(const float* x, int64_t T, int64_t d, float eps, uint16_t* xo, moe_stream_t stream) {
    if (!x || !xo || T < 0 || d < 1 || d > kMaxDim) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    return cuda_status(launch_rmsnorm_bf16(x, T, d, eps, xo, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_get_device_status(void* workspace, moe_stream_t stream, int32_t* device_code) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t code = 0;
    cudaError_t e = cudaMemcpyAsync(&code, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && code != 0) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (device_code) *device_code = code;
    return code == 0 ? MOE_OK : MOE_ERR_DEVICE_CHECK;
}

}  // extern "C"
