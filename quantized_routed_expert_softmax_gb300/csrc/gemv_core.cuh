// gemv_core.cuh -- the weight-streaming GEMV core shared by the expert kernels
// (gemv.cu) and the one-kernel decode layer (decode.cu): streaming loads and per-thread
// asynchronous copies, exact code -> f16 conversions, and the tensor-core panel product
// (mma.sync m16n8k16, f16 inputs, f32 accumulation) over the K-panel weight layout.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Same, with an L2 evict-first policy: weights read once should not push out data that
// is still wanted (the down weights prefetched into L2 while gate.up streams).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint4 ldg_stream16_ef(const uint8_t* p, uint64_t pol) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol));
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

__device__ __forceinline__ uint32_t ldg_u16(const uint8_t* p) {
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Bring `bytes` (a multiple of 16, 16-byte aligned) into L2 without loading registers.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Per-thread asynchronous copies global -> shared (no registers held while in flight).
__device__ __forceinline__ void cp_async16_ef(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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
__device__ __forceinline__ void load_token_rows(const ExpertArgs& a, const int4& si, int t0, int nt, float* xs) {
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
        *reinterpret_cast<float4*>(xs + t * a.d + c) = v;
    }
}

__device__ __forceinline__ void load_h_rows(const ExpertArgs& a, int r0, int t0, int nt, float* hs) {
    const int f4 = a.f / 4;
    const float4* src = reinterpret_cast<const float4*>(a.ws.h + static_cast<int64_t>(r0 + t0) * a.f);
    for (int i = threadIdx.x; i < nt * f4; i += blockDim.x) reinterpret_cast<float4*>(hs)[i] = __ldcg(src + i);
}

// ------------------------------------------------------------------------------ tensor-core GEMV core
// The multiply-adds run on the tensor cores (mma.sync m16n8k16, f16 inputs, f32
// accumulation) so the only per-weight ALU work is the exact conversion of the code to f16:
//   Q8_0 : byte-insert the (sign-flipped) int8 into the mantissa of 1024.0h and subtract
//          1152.0h: exact integers -128..127; the fp16 block scale is applied to the f32
//          result of each 32-column panel;
//   NVFP4: cvt.rn.f16x2.e2m1x2, times the E4M3 block scale (exact: 2 x 4 significant bits).
// A warp computes two 16-row blocks (A, B) of a 32-row tile over its share of the K panels;
// up to 8 tokens ride in the MMA's N = 8 columns for free.  In the K order of the MMA,
// thread t of a quad owns 8 (Q8_0) or 16 (NVFP4) consecutive columns of a panel, the same
// columns for the weights (A) and the activations (B), so any assignment is a valid dot
// product order.
//
// A warp streams its panels through a ring of kStages slots in shared memory: per slot the
// 2 x 512 code bytes of its 32 rows and their scales (64 or 128 bytes), copied with
// cp.async by all 32 lanes; cp.async.wait_group + __syncwarp make a slot readable.
constexpr int kStages = 6;
constexpr int kSlotBytes = 1024 + 128;

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four signed int8 in a word -> two f16x2 (bytes 0,1 and bytes 2,3), exact.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;                       // int8 + 128 as unsigned bytes
    const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);   // halves 0x64 u0, 0x64 u1 = 1024 + u
    const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    const __half2 lv = __hsub2(*reinterpret_cast<const __half2*>(&l), off);
    const __half2 hv = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
    lo = *reinterpret_cast<const uint32_t*>(&lv);
    hi = *reinterpret_cast<const uint32_t*>(&hv);
}

// One byte of two E2M1 codes times an f16 scale -> f16x2, exact.
__device__ __forceinline__ uint32_t e2m1x2_scaled(uint32_t byte, __half2 sc) {
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
    const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&h2), sc);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ __half2 e4m3_to_h2(uint32_t byte) {
    uint32_t h2;
    const uint16_t in = static_cast<uint16_t>(byte & 0xffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    const __half h = __ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu));
    return __halves2half2(h, h);
}

// Copy one panel's codes of rows [rowA, rowA+16) and [rowB, rowB+16) and their scales into
// a slot.  Chunk c (16 bytes) of a 512-byte block is row c/2, columns 16*(c%2)..; `skip`
// bit 0 / 1 drops the first / second 16 columns (inactive neuron groups, Q8_0 down).
// Per-channel int8 (MOE_W_INT8PC, device layout): the rows' fp32 scales first, then panels
// of 32 codes per row; every panel of a row tile copies the same 2 x 64 bytes of scales.
template <int FMT>
__device__ __forceinline__ void issue_panel_block(uint32_t slot, const uint8_t* W, int rows, int rowA, int rowB,
                                                  int b, uint64_t pol, int skip) {
    const int lane = threadIdx.x & 31;
    if (FMT == MOE_W_INT8PC) {
        const uint8_t* P = W + static_cast<int64_t>(rows) * 4 + static_cast<int64_t>(b) * rows * 32;
        if (!((skip >> (lane & 1)) & 1)) {
            cp_async16_ef(slot + lane * 16, P + rowA * 32 + lane * 16, pol);
            cp_async16_ef(slot + 512 + lane * 16, P + rowB * 32 + lane * 16, pol);
        }
        if (lane < 4) cp_async16(slot + 1024 + lane * 16, W + rowA * 4 + lane * 16);
        else if (lane < 8) cp_async16(slot + 1024 + 64 + (lane - 4) * 16, W + rowB * 4 + (lane - 4) * 16);
        return;
    }
    const int64_t pbytes = static_cast<int64_t>(rows) * (FMT == MOE_W_Q8_0 ? 34 : 36);
    const uint8_t* P = W + b * pbytes;
    const bool keep = !((skip >> (lane & 1)) & 1);
    if (keep) {
        cp_async16_ef(slot + lane * 16, P + rowA * 32 + lane * 16, pol);
        cp_async16_ef(slot + 512 + lane * 16, P + rowB * 32 + lane * 16, pol);
    }
    const uint8_t* S = P + rows * 32;
    if (FMT == MOE_W_Q8_0) {   // 2 bytes per row: 32 bytes per block
        if (lane < 2) cp_async16(slot + 1024 + lane * 16, S + rowA * 2 + lane * 16);
        else if (lane < 4) cp_async16(slot + 1024 + 32 + (lane - 2) * 16, S + rowB * 2 + (lane - 2) * 16);
    } else {                   // 4 bytes per row: 64 bytes per block
        if (lane < 4) cp_async16(slot + 1024 + lane * 16, S + rowA * 4 + lane * 16);
        else if (lane < 8) cp_async16(slot + 1024 + 64 + (lane - 4) * 16, S + rowB * 4 + (lane - 4) * 16);
    }
}

// acc[blk][i] += this panel's contribution; xs: f16 activations [8 tokens][ld] (rows >= nt
// are never read: their B fragments are zero).  `skip`: inactive 16-column halves.
// With `split`, the activations are fp32 values carried as two f16 terms (hi at xs, lo at
// xs + lo_off, v ~= hi + lo to ~22 bits): each weight fragment meets both.
template <int FMT>
__device__ __forceinline__ void panel_mma(const unsigned char* slot, const __half* xs, int ld, int b, int nt,
                                          int skip, float acc[2][4], bool split, int lo_off) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const bool has_tok = g < nt;
    if (FMT == MOE_W_Q8_0 || FMT == MOE_W_INT8PC) {
        uint4 xv = make_uint4(0, 0, 0, 0), xl = make_uint4(0, 0, 0, 0);
        if (has_tok) {
            xv = *reinterpret_cast<const uint4*>(xs + g * ld + b * 32 + 8 * t);
            if (split) xl = *reinterpret_cast<const uint4*>(xs + lo_off + g * ld + b * 32 + 8 * t);
        }
        const bool dead = (skip >> (t >> 1)) & 1;   // thread t covers columns 8t..8t+7
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            const unsigned char* cb = slot + blk * 512;
            uint2 r0 = *reinterpret_cast<const uint2*>(cb + g * 32 + 8 * t);
            uint2 r8 = *reinterpret_cast<const uint2*>(cb + (g + 8) * 32 + 8 * t);
            if (dead) r0 = r8 = make_uint2(0u, 0u);   // a skipped group: its bytes were not copied
            float s0, s8;   // Q8_0: the block's fp16 scales; per-channel int8: the rows' fp32 scales
            if (FMT == MOE_W_Q8_0) {
                const unsigned short* sc = reinterpret_cast<const unsigned short*>(slot + 1024 + blk * 32);
                s0 = __half2float(__ushort_as_half(sc[g]));
                s8 = __half2float(__ushort_as_half(sc[g + 8]));
            } else {
                const float* sc = reinterpret_cast<const float*>(slot + 1024 + blk * 64);
                s0 = sc[g];
                s8 = sc[g + 8];
            }
            uint32_t a0, a2, a1, a3, c0, c2, c1, c3;
            s8x4_to_f16x2x2(r0.x, a0, a2);
            s8x4_to_f16x2x2(r8.x, a1, a3);
            s8x4_to_f16x2x2(r0.y, c0, c2);
            s8x4_to_f16x2x2(r8.y, c1, c3);
            float dd[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(dd, a0, a1, a2, a3, xv.x, xv.y);
            mma16816(dd, c0, c1, c2, c3, xv.z, xv.w);
            if (split) {
                mma16816(dd, a0, a1, a2, a3, xl.x, xl.y);
                mma16816(dd, c0, c1, c2, c3, xl.z, xl.w);
            }
            acc[blk][0] = fmaf(s0, dd[0], acc[blk][0]);
            acc[blk][1] = fmaf(s0, dd[1], acc[blk][1]);
            acc[blk][2] = fmaf(s8, dd[2], acc[blk][2]);
            acc[blk][3] = fmaf(s8, dd[3], acc[blk][3]);
        }
    } else {
        uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
        uint4 l0 = make_uint4(0, 0, 0, 0), l1 = make_uint4(0, 0, 0, 0);
        if (has_tok) {
            x0 = *reinterpret_cast<const uint4*>(xs + g * ld + b * 64 + 16 * t);
            x1 = *reinterpret_cast<const uint4*>(xs + g * ld + b * 64 + 16 * t + 8);
            if (split) {
                l0 = *reinterpret_cast<const uint4*>(xs + lo_off + g * ld + b * 64 + 16 * t);
                l1 = *reinterpret_cast<const uint4*>(xs + lo_off + g * ld + b * 64 + 16 * t + 8);
            }
        }
        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t xlw[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            const unsigned char* cb = slot + blk * 512;
            const uint2 r0 = *reinterpret_cast<const uint2*>(cb + g * 32 + 8 * t);
            const uint2 r8 = *reinterpret_cast<const uint2*>(cb + (g + 8) * 32 + 8 * t);
            const unsigned char* sc = slot + 1024 + blk * 64;   // 4 scale bytes per row
            const __half2 s0 = e4m3_to_h2(sc[g * 4 + t]);         // columns 16t.. are sub-block t
            const __half2 s8 = e4m3_to_h2(sc[(g + 8) * 4 + t]);
#pragma unroll
            for (int m = 0; m < 4; ++m) {   // 4 MMAs of 16 columns: bytes 2m, 2m+1 of the 8
                const uint32_t w0 = (m < 2) ? r0.x : r0.y;
                const uint32_t w8 = (m < 2) ? r8.x : r8.y;
                const int sh = (m & 1) * 16;
                const uint32_t a0 = e2m1x2_scaled((w0 >> sh) & 0xffu, s0);
                const uint32_t a2 = e2m1x2_scaled((w0 >> (sh + 8)) & 0xffu, s0);
                const uint32_t a1 = e2m1x2_scaled((w8 >> sh) & 0xffu, s8);
                const uint32_t a3 = e2m1x2_scaled((w8 >> (sh + 8)) & 0xffu, s8);
                mma16816(acc[blk], a0, a1, a2, a3, xw[2 * m], xw[2 * m + 1]);
                if (split) mma16816(acc[blk], a0, a1, a2, a3, xlw[2 * m], xlw[2 * m + 1]);
            }
        }
    }
}

// v ~= hi + lo with both terms f16 (lo = f16(v - hi)).
__device__ __forceinline__ void split_f16(float v0, float v1, __half2& hi, __half2& lo) {
    hi = __floats2half2_rn(v0, v1);
    const float2 h = __half22float2(hi);
    lo = __floats2half2_rn(v0 - h.x, v1 - h.y);
}

}  // namespace moe
