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
// Layout in HBM (see include/moe.h): weights in K panels, so that lane l of a warp owns
// one weight row and streams it 32 bytes per panel; a warp reads 1 KB contiguous per
// panel (fully coalesced) and no cross-lane reduction is needed.  The tokens of one
// expert sit in shared memory as fp32; dequantisation is exact (int8 or e2m1 codes
// times the block scale) and accumulation is fp32.  One CTA's 8 warps split the K
// panels of its rows and reduce through shared memory in a fixed order, so results are
// bitwise reproducible.
#include "common.cuh"

namespace moe {


__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream4(const uint8_t* p) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const uint8_t* p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ float ldg_half(const uint8_t* p) {
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return __half2float(__ushort_as_half(v));
}

__device__ __forceinline__ uint32_t word_of(const uint4& a, const uint4& b, int i) {
    switch (i) {
        case 0: return a.x;
        case 1: return a.y;
        case 2: return a.z;
        case 3: return a.w;
        case 4: return b.x;
        case 5: return b.y;
        case 6: return b.z;
        default: return b.w;
    }
}

__device__ __forceinline__ float f4get(const float4& v, int j) {
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// Load the x rows of `nt` tokens (sorted rows r0+t0 ...) into shared memory as fp32.
__device__ __forceinline__ void load_token_rows(const ExpertArgs& a, int r0, int t0, int nt, float* xs) {
    const int d4 = a.d / 4;
    for (int i = threadIdx.x; i < nt * d4; i += blockDim.x) {
        const int t = i / d4, c = (i % d4) * 4;
        const int pair = a.ws.perm[r0 + t0 + t];
        const int64_t off = static_cast<int64_t>(pair / a.k) * a.d + c;
        float4 v;
        if (a.xt == MOE_F32) {
            v = *reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + off);
        } else {
            const uint2 b = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.x) + off);
            v = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u),
                            __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u));
        }
        *reinterpret_cast<float4*>(xs + t * a.d + c) = v;
    }
}

// ------------------------------------------------------------------------------ gate.up
// Partial dot products of this lane's weight row with N tokens over panels [pb, pe).
template <int FMT, int N>
__device__ __forceinline__ void gu_dot(const ExpertArgs& a, const uint8_t* W, int row, int pb, int pe,
                                       const float* xs, float acc[N]) {
    const int rows = a.rows_gu;
    const int d = a.d;
    constexpr int U = 4;
    if (FMT == MOE_W_Q8_0) {
        const int64_t pbytes = static_cast<int64_t>(rows) * 34;
        for (int b = pb; b < pe; b += U) {
            uint4 q0[U], q1[U];
            float sc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (b + u < pe) {
                    const uint8_t* P = W + (b + u) * pbytes;
                    q0[u] = ldg_stream16(P + row * 32);
                    q1[u] = ldg_stream16(P + row * 32 + 16);
                    sc[u] = ldg_half(P + rows * 32 + row * 2);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (b + u < pe) {
                    float part[N];
#pragma unroll
                    for (int t = 0; t < N; ++t) part[t] = 0.0f;
                    const float* xb = xs + (b + u) * 32;
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {
                        const uint32_t word = word_of(q0[u], q1[u], wi);
                        float4 xv[N];
#pragma unroll
                        for (int t = 0; t < N; ++t) xv[t] = *reinterpret_cast<const float4*>(xb + t * d + wi * 4);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float v = s8_to_f32(word, j);
#pragma unroll
                            for (int t = 0; t < N; ++t) part[t] = fmaf(v, f4get(xv[t], j), part[t]);
                        }
                    }
#pragma unroll
                    for (int t = 0; t < N; ++t) acc[t] = fmaf(sc[u], part[t], acc[t]);
                }
            }
        }
    } else {   // NVFP4, panels of 64 columns: 32 code bytes + 4 scale bytes per row
        const int64_t pbytes = static_cast<int64_t>(rows) * 36;
        for (int b = pb; b < pe; b += U) {
            uint4 q0[U], q1[U];
            uint32_t sw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (b + u < pe) {
                    const uint8_t* P = W + (b + u) * pbytes;
                    q0[u] = ldg_stream16(P + row * 32);
                    q1[u] = ldg_stream16(P + row * 32 + 16);
                    sw[u] = ldg_stream4(P + rows * 32 + row * 4);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (b + u < pe) {
                    const float* xb = xs + (b + u) * 64;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {      // 4 sub-blocks of 16 values
                        float part[N];
#pragma unroll
                        for (int t = 0; t < N; ++t) part[t] = 0.0f;
#pragma unroll
                        for (int wi = 0; wi < 2; ++wi) {
                            const uint32_t word = word_of(q0[u], q1[u], 2 * s + wi);
#pragma unroll
                            for (int by = 0; by < 4; ++by) {
                                const float2 v = e2m1x2_to_f32x2((word >> (8 * by)) & 0xffu);
                                const int c = 16 * s + 8 * wi + 2 * by;
#pragma unroll
                                for (int t = 0; t < N; ++t) {
                                    const float2 xv = *reinterpret_cast<const float2*>(xb + t * d + c);
                                    part[t] = fmaf(v.x, xv.x, part[t]);
                                    part[t] = fmaf(v.y, xv.y, part[t]);
                                }
                            }
                        }
                        const float sb = e4m3_to_f32((sw[u] >> (8 * s)) & 0xffu);
#pragma unroll
                        for (int t = 0; t < N; ++t) acc[t] = fmaf(sb, part[t], acc[t]);
                    }
                }
            }
        }
    }
}

template <int FMT, int ACT, int N>
__device__ __forceinline__ void gu_tile(const ExpertArgs& a, const uint8_t* W, int row, int pb, int pe,
                                        const float* xs, float (*red)[8][32], int e, int r0, int t0, int nt,
                                        int tile, uint32_t* act_bits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float acc[N];
#pragma unroll
    for (int t = 0; t < N; ++t) acc[t] = 0.0f;
    gu_dot<FMT, N>(a, W, row, pb, pe, xs, acc);
#pragma unroll
    for (int t = 0; t < N; ++t) red[warp][t][lane] = acc[t];
    __syncthreads();
    if (warp < nt) {
        const int t = warp;
        float z = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) z += red[w][t][lane];
        if (FMT == MOE_W_NVFP4) z *= a.gu_ts[e];
        float* hrow = a.ws.h + static_cast<int64_t>(r0 + t0 + t) * a.f;
        if (ACT == MOE_ACT_SWIGLU) {
            const float u = __shfl_down_sync(0xffffffffu, z, 16);
            const float h = silu(z) * u;
            if (lane < 16) hrow[tile * 16 + lane] = h;
            const uint32_t nz = __ballot_sync(0xffffffffu, lane < 16 && h != 0.0f);
            if (lane == 0 && nz) atomicOr(act_bits, 1u);
        } else {
            const float h = z > 0.0f ? z * z : 0.0f;
            hrow[tile * 32 + lane] = h;
            const uint32_t nz = __ballot_sync(0xffffffffu, h != 0.0f);
            if (lane == 0 && nz) atomicOr(act_bits, ((nz & 0xffffu) ? 1u : 0u) | ((nz >> 16) ? 2u : 0u));
        }
    }
}

// grid: (f/16 tiles for SwiGLU or f/32 for ReLU^2, active-slot capacity); block 256.
// TT: the largest token tile this launch needs (1, 2, 4 or 8); smaller tiles of the same
// launch use the narrower bodies, so a one-token launch carries no wide accumulators.
template <int FMT, int ACT, int TT>
__global__ void __launch_bounds__(256) gate_up_gemv_kernel(ExpertArgs a) {
    const int slot = blockIdx.y;
    if (slot >= *a.ws.n_active) return;
    const int e = a.ws.act_e[slot];
    const int r0 = a.ws.offsets[e];
    const int cnt = a.ws.offsets[e + 1] - r0;
    extern __shared__ __align__(16) float xs[];
    __shared__ float red[8][8][32];
    __shared__ uint32_t act_bits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x;
    const int row = (ACT == MOE_ACT_SWIGLU) ? (lane < 16 ? tile * 16 + lane : a.f + tile * 16 + lane - 16)
                                            : tile * 32 + lane;
    const uint8_t* W = a.w_gu + static_cast<int64_t>(e) * a.gu_bytes;
    const int npan = (FMT == MOE_W_Q8_0) ? a.d / 32 : a.d / 64;
    const int pb = warp * npan / 8, pe = (warp + 1) * npan / 8;
    if (threadIdx.x == 0) act_bits = 0;
    for (int t0 = 0; t0 < cnt; t0 += a.tt_gu) {
        const int nt = min(a.tt_gu, cnt - t0);
        __syncthreads();
        load_token_rows(a, r0, t0, nt, xs);
        __syncthreads();
        if (TT == 1 || nt == 1) gu_tile<FMT, ACT, 1>(a, W, row, pb, pe, xs, red, e, r0, t0, nt, tile, &act_bits);
        else if (TT == 2 || nt == 2) gu_tile<FMT, ACT, (TT < 2 ? TT : 2)>(a, W, row, pb, pe, xs, red, e, r0, t0, nt, tile, &act_bits);
        else if (TT == 4 || nt <= 4) gu_tile<FMT, ACT, (TT < 4 ? TT : 4)>(a, W, row, pb, pe, xs, red, e, r0, t0, nt, tile, &act_bits);
        else gu_tile<FMT, ACT, TT>(a, W, row, pb, pe, xs, red, e, r0, t0, nt, tile, &act_bits);
    }
    __syncthreads();
    if (threadIdx.x == 0 && act_bits) {
        const int g0 = (ACT == MOE_ACT_SWIGLU) ? tile : 2 * tile;
        uint32_t bits = (ACT == MOE_ACT_SWIGLU) ? 1u : act_bits;
        atomicOr(a.ws.gmask + slot * a.gwords + g0 / 32, bits << (g0 % 32));
    }
}

// ------------------------------------------------------------------------------ down, Q8_0
// Q8_0 down matrices [d][f] in K panels of 32 neurons.  Lane = one output row; a panel
// holds neuron groups 2b and 2b+1 and each 16-byte half is read only if its group is
// active.  grid: (d/256, slot capacity, ksplit); block 256 (8 warps x 32 rows).
template <int N>
__device__ __forceinline__ void dn_q8_tile(const ExpertArgs& a, const uint8_t* W, int row, int pb, int pe,
                                           const float* hs, const uint32_t* gm, float acc[N]) {
    const int d = a.d, f = a.f;
    const int64_t pbytes = static_cast<int64_t>(d) * 34;
    constexpr int U = 4;
    for (int b = pb; b < pe; b += U) {
        uint4 q0[U], q1[U];
        float sc[U];
        bool a0[U], a1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            a0[u] = a1[u] = false;
            if (b + u < pe) {
                const int g = 2 * (b + u);
                a0[u] = (gm[g >> 5] >> (g & 31)) & 1u;
                a1[u] = (gm[(g + 1) >> 5] >> ((g + 1) & 31)) & 1u;
                const uint8_t* P = W + (b + u) * pbytes;
                q0[u] = a0[u] ? ldg_stream16(P + row * 32) : make_uint4(0, 0, 0, 0);
                q1[u] = a1[u] ? ldg_stream16(P + row * 32 + 16) : make_uint4(0, 0, 0, 0);
                sc[u] = (a0[u] || a1[u]) ? ldg_half(P + d * 32 + row * 2) : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (b + u < pe && (a0[u] || a1[u])) {
                float part[N];
#pragma unroll
                for (int t = 0; t < N; ++t) part[t] = 0.0f;
                const float* hb = hs + (b + u) * 32;
#pragma unroll
                for (int wi = 0; wi < 8; ++wi) {
                    if ((wi < 4 && !a0[u]) || (wi >= 4 && !a1[u])) continue;
                    const uint32_t word = word_of(q0[u], q1[u], wi);
                    float4 hv[N];
#pragma unroll
                    for (int t = 0; t < N; ++t) hv[t] = *reinterpret_cast<const float4*>(hb + t * f + wi * 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float v = s8_to_f32(word, j);
#pragma unroll
                        for (int t = 0; t < N; ++t) part[t] = fmaf(v, f4get(hv[t], j), part[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < N; ++t) acc[t] = fmaf(sc[u], part[t], acc[t]);
            }
        }
    }
}

__device__ __forceinline__ void load_h_rows(const ExpertArgs& a, int r0, int t0, int nt, float* hs) {
    const int f4 = a.f / 4;
    const float4* src = reinterpret_cast<const float4*>(a.ws.h + static_cast<int64_t>(r0 + t0) * a.f);
    for (int i = threadIdx.x; i < nt * f4; i += blockDim.x) reinterpret_cast<float4*>(hs)[i] = src[i];
}

template <int TT>
__global__ void __launch_bounds__(256) down_q8_gemv_kernel(ExpertArgs a) {
    const int slot = blockIdx.y;
    if (slot >= *a.ws.n_active) return;
    const int e = a.ws.act_e[slot];
    const int r0 = a.ws.offsets[e];
    const int cnt = a.ws.offsets[e + 1] - r0;
    extern __shared__ __align__(16) float hs[];
    __shared__ uint32_t gm[64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 256 + warp * 32 + lane;
    const int npan = a.f / 32;
    const int z = blockIdx.z;
    const int pb = z * npan / a.ksplit, pe = (z + 1) * npan / a.ksplit;
    const uint8_t* W = a.w_dn + static_cast<int64_t>(e) * a.dn_bytes;
    for (int i = threadIdx.x; i < a.gwords; i += blockDim.x) gm[i] = a.ws.gmask[slot * a.gwords + i];
    float* ybase = a.ws.y + static_cast<int64_t>(z) * a.P * a.d;
    for (int t0 = 0; t0 < cnt; t0 += a.tt_dn) {
        const int nt = min(a.tt_dn, cnt - t0);
        __syncthreads();
        load_h_rows(a, r0, t0, nt, hs);
        __syncthreads();
#define MOE_DN_Q8_CASE(NN)                                                              \
    {                                                                                   \
        float acc[NN];                                                                  \
        _Pragma("unroll") for (int t = 0; t < NN; ++t) acc[t] = 0.0f;                   \
        dn_q8_tile<NN>(a, W, row, pb, pe, hs, gm, acc);                                 \
        _Pragma("unroll") for (int t = 0; t < NN; ++t) if (t < nt)                      \
            ybase[static_cast<int64_t>(r0 + t0 + t) * a.d + row] = acc[t];              \
    }
        if (TT == 1 || nt == 1) MOE_DN_Q8_CASE(1)
        else if (TT == 2 || nt == 2) MOE_DN_Q8_CASE((TT < 2 ? TT : 2))
        else if (TT == 4 || nt <= 4) MOE_DN_Q8_CASE((TT < 4 ? TT : 4))
        else MOE_DN_Q8_CASE(TT)
#undef MOE_DN_Q8_CASE
    }
}

// ------------------------------------------------------------------------------ down, NVFP4
// NVFP4 down matrices in the neuron layout: per group of 16 neurons, each neuron's codes
// for all d rows (d/2 bytes), then the d scale bytes.  A warp covers 256 rows: lane l
// rows 256*rt + 8l .. +7 (4 code bytes per neuron, 8 scale bytes).  Inactive groups are
// not read at all.  grid: (ceil(d/1024), slot capacity, ksplit); block 128 (4 row tiles).
template <int N>
__device__ __forceinline__ void dn_nv_tile(const ExpertArgs& a, const uint8_t* W, int rt, int gb, int ge,
                                           const float* hs, const uint32_t* gm, float acc[N][8]) {
    const int d = a.d, f = a.f;
    const int lane = threadIdx.x & 31;
    const int64_t rec = 16 * (d / 2) + d;
    for (int g = gb; g < ge; ++g) {
        if (!((gm[g >> 5] >> (g & 31)) & 1u)) continue;
        const uint8_t* base = W + g * rec;
        uint32_t codes[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) codes[j] = ldg_stream4(base + j * (d / 2) + rt * 128 + lane * 4);
        const uint2 sc = ldg_stream8(base + 16 * (d / 2) + rt * 256 + lane * 8);
        float part[N][8];
#pragma unroll
        for (int t = 0; t < N; ++t)
#pragma unroll
            for (int r = 0; r < 8; ++r) part[t][r] = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float hv[N];
#pragma unroll
            for (int t = 0; t < N; ++t) hv[t] = hs[t * f + 16 * g + j];
#pragma unroll
            for (int by = 0; by < 4; ++by) {
                const float2 v = e2m1x2_to_f32x2((codes[j] >> (8 * by)) & 0xffu);   // rows 2by, 2by+1
#pragma unroll
                for (int t = 0; t < N; ++t) {
                    part[t][2 * by] = fmaf(v.x, hv[t], part[t][2 * by]);
                    part[t][2 * by + 1] = fmaf(v.y, hv[t], part[t][2 * by + 1]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float sb = e4m3_to_f32(((r < 4 ? sc.x : sc.y) >> (8 * (r & 3))) & 0xffu);
#pragma unroll
            for (int t = 0; t < N; ++t) acc[t][r] = fmaf(sb, part[t][r], acc[t][r]);
        }
    }
}

template <int TT>
__global__ void __launch_bounds__(128) down_nv_gemv_kernel(ExpertArgs a) {
    const int slot = blockIdx.y;
    if (slot >= *a.ws.n_active) return;
    const int e = a.ws.act_e[slot];
    const int r0 = a.ws.offsets[e];
    const int cnt = a.ws.offsets[e + 1] - r0;
    extern __shared__ __align__(16) float hs[];
    __shared__ uint32_t gm[64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rt = blockIdx.x * 4 + warp;            // row tile of this warp
    const bool has_rows = rt < a.d / 256;
    const int ng = a.f / 16;
    const int z = blockIdx.z;
    const int gb = z * ng / a.ksplit, ge = (z + 1) * ng / a.ksplit;
    const uint8_t* W = a.w_dn + static_cast<int64_t>(e) * a.dn_bytes;
    const float ts = a.dn_ts[e];
    for (int i = threadIdx.x; i < a.gwords; i += blockDim.x) gm[i] = a.ws.gmask[slot * a.gwords + i];
    float* ybase = a.ws.y + static_cast<int64_t>(z) * a.P * a.d;
    const int row0 = rt * 256 + lane * 8;
    for (int t0 = 0; t0 < cnt; t0 += a.tt_dn) {
        const int nt = min(a.tt_dn, cnt - t0);
        __syncthreads();
        load_h_rows(a, r0, t0, nt, hs);
        __syncthreads();
        if (!has_rows) continue;
#define MOE_DN_NV_CASE(NN)                                                                      \
    {                                                                                           \
        float acc[NN][8];                                                                       \
        _Pragma("unroll") for (int t = 0; t < NN; ++t) _Pragma("unroll") for (int r = 0; r < 8; ++r) \
            acc[t][r] = 0.0f;                                                                   \
        dn_nv_tile<NN>(a, W, rt, gb, ge, hs, gm, acc);                                          \
        _Pragma("unroll") for (int t = 0; t < NN; ++t) if (t < nt) {                            \
            float* yr = ybase + static_cast<int64_t>(r0 + t0 + t) * a.d + row0;                 \
            *reinterpret_cast<float4*>(yr) =                                                    \
                make_float4(acc[t][0] * ts, acc[t][1] * ts, acc[t][2] * ts, acc[t][3] * ts);    \
            *reinterpret_cast<float4*>(yr + 4) =                                                \
                make_float4(acc[t][4] * ts, acc[t][5] * ts, acc[t][6] * ts, acc[t][7] * ts);    \
        }                                                                                       \
    }
        if (TT == 1 || nt == 1) MOE_DN_NV_CASE(1)
        else if (TT == 2 || nt == 2) MOE_DN_NV_CASE((TT < 2 ? TT : 2))
        else MOE_DN_NV_CASE((TT < 4 ? TT : 4))
#undef MOE_DN_NV_CASE
    }
}

// ------------------------------------------------------------------------------ combine
// out[t] = sum_{j<k} w[t][j] * sum_{z<ksplit} y[z][pos(t,j)], both sums in index order.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ w, const int32_t* __restrict__ pos,
                                                       const float* __restrict__ y, int k, int d, int ksplit,
                                                       int64_t zstride, float* __restrict__ out) {
    const int t = blockIdx.y;
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (c >= d) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int r = pos[t * k + j];
        const float wt = w[t * k + j];
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int z = 0; z < ksplit; ++z) {
            const float4 v = *reinterpret_cast<const float4*>(y + z * zstride + static_cast<int64_t>(r) * d + c);
            s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
        }
        acc.x = fmaf(wt, s.x, acc.x);
        acc.y = fmaf(wt, s.y, acc.y);
        acc.z = fmaf(wt, s.z, acc.z);
        acc.w = fmaf(wt, s.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + static_cast<int64_t>(t) * d + c) = acc;
}

// ------------------------------------------------------------------------------ rmsnorm glue
__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float* __restrict__ x, int d, float eps,
                                                            uint16_t* __restrict__ xo) {
    const int t = blockIdx.x;
    const float* xr = x + static_cast<int64_t>(t) * d;
    float ss = 0.0f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
    ss = warp_sum(ss);
    __shared__ float ws[8];
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += ws[i];
    const float inv = rsqrtf(tot / static_cast<float>(d) + eps);
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        xo[static_cast<int64_t>(t) * d + i] = __bfloat16_as_ushort(__float2bfloat16_rn(xr[i] * inv));
}

// ------------------------------------------------------------------------------ launchers
template <typename K>
static cudaError_t allow_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int FMT, int ACT, int TT>
static cudaError_t gu_launch(const ExpertArgs& a, dim3 grid, size_t smem, cudaStream_t s, bool configure) {
    if (configure) return allow_smem(gate_up_gemv_kernel<FMT, ACT, TT>, 200 * 1024);
    gate_up_gemv_kernel<FMT, ACT, TT><<<grid, 256, smem, s>>>(a);
    return cudaGetLastError();
}

template <int FMT, int ACT>
static cudaError_t gu_dispatch_tt(const ExpertArgs& a, dim3 grid, size_t smem, cudaStream_t s, bool configure) {
    switch (a.tt_gu) {
        case 1: return gu_launch<FMT, ACT, 1>(a, grid, smem, s, configure);
        case 2: return gu_launch<FMT, ACT, 2>(a, grid, smem, s, configure);
        case 4: return gu_launch<FMT, ACT, 4>(a, grid, smem, s, configure);
        default: return gu_launch<FMT, ACT, 8>(a, grid, smem, s, configure);
    }
}

static cudaError_t gu_dispatch(const ExpertArgs& a, int wfmt, int act, dim3 grid, size_t smem, cudaStream_t s,
                               bool configure) {
    if (wfmt == MOE_W_Q8_0 && act == MOE_ACT_SWIGLU)
        return gu_dispatch_tt<MOE_W_Q8_0, MOE_ACT_SWIGLU>(a, grid, smem, s, configure);
    if (wfmt == MOE_W_Q8_0) return gu_dispatch_tt<MOE_W_Q8_0, MOE_ACT_RELU2>(a, grid, smem, s, configure);
    if (act == MOE_ACT_SWIGLU) return gu_dispatch_tt<MOE_W_NVFP4, MOE_ACT_SWIGLU>(a, grid, smem, s, configure);
    return gu_dispatch_tt<MOE_W_NVFP4, MOE_ACT_RELU2>(a, grid, smem, s, configure);
}

template <int TT>
static cudaError_t dn_launch(const ExpertArgs& a, int wfmt, int slot_cap, size_t smem, cudaStream_t s,
                             bool configure) {
    if (wfmt == MOE_W_Q8_0) {
        if (configure) return allow_smem(down_q8_gemv_kernel<TT>, 200 * 1024);
        down_q8_gemv_kernel<TT><<<dim3(a.d / 256, slot_cap, a.ksplit), 256, smem, s>>>(a);
    } else {
        if (configure) return allow_smem(down_nv_gemv_kernel<(TT < 4 ? TT : 4)>, 200 * 1024);
        down_nv_gemv_kernel<(TT < 4 ? TT : 4)><<<dim3((a.d / 256 + 3) / 4, slot_cap, a.ksplit), 128, smem, s>>>(a);
    }
    return cudaGetLastError();
}

static cudaError_t dn_dispatch(const ExpertArgs& a, int wfmt, int slot_cap, size_t smem, cudaStream_t s,
                               bool configure) {
    switch (a.tt_dn) {
        case 1: return dn_launch<1>(a, wfmt, slot_cap, smem, s, configure);
        case 2: return dn_launch<2>(a, wfmt, slot_cap, smem, s, configure);
        case 4: return dn_launch<4>(a, wfmt, slot_cap, smem, s, configure);
        default: return dn_launch<8>(a, wfmt, slot_cap, smem, s, configure);
    }
}

// Raise the dynamic shared-memory limit of every expert-kernel instantiation (once per
// device).
cudaError_t configure_gemv_kernels() {
    ExpertArgs a{};
    const int wf[2] = {MOE_W_Q8_0, MOE_W_NVFP4};
    const int ac[2] = {MOE_ACT_SWIGLU, MOE_ACT_RELU2};
    const int tts[4] = {1, 2, 4, 8};
    for (int tt : tts) {
        a.tt_gu = a.tt_dn = tt;
        for (int w : wf) {
            for (int c : ac) {
                cudaError_t e = gu_dispatch(a, w, c, dim3(1), 0, nullptr, true);
                if (e != cudaSuccess) return e;
            }
            cudaError_t e = dn_dispatch(a, w, 1, 0, nullptr, true);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_gate_up_gemv(const ExpertArgs& a, int wfmt, int act, int slot_cap, cudaStream_t s) {
    const int tiles = (act == MOE_ACT_SWIGLU) ? a.f / 16 : a.f / 32;
    const size_t smem = static_cast<size_t>(a.tt_gu) * a.d * sizeof(float);
    return gu_dispatch(a, wfmt, act, dim3(tiles, slot_cap), smem, s, false);
}

cudaError_t launch_down_gemv(const ExpertArgs& a, int wfmt, int slot_cap, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(a.tt_dn) * a.f * sizeof(float);
    return dn_dispatch(a, wfmt, slot_cap, smem, s, false);
}

cudaError_t launch_combine(const float* w, const int32_t* pos, const float* y, int64_t T, int k, int64_t d,
                           int ksplit, int64_t zstride, float* out, cudaStream_t s) {
    const int64_t cols4 = d / 4;
    const dim3 grid(static_cast<unsigned>((cols4 + 255) / 256), static_cast<unsigned>(T));
    combine_kernel<<<grid, 256, 0, s>>>(w, pos, y, k, (int)d, ksplit, zstride, out);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const float* x, int64_t T, int64_t d, float eps, uint16_t* xo, cudaStream_t s) {
    rmsnorm_bf16_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(x, (int)d, eps, xo);
    return cudaGetLastError();
}

}  // namespace moe
