// pack.cu -- weight packers: Q8_0 and NVFP4 (with the neuron-contiguous down relayout).
//
// Q8_0: 32 int8 codes + one fp16 scale per block of 32 along a row; d = amax/127,
// codes = round-half-away(x * (1/d)) with the fp32 d (the Q8_0 experts of "Running Gemma
// 4 26B at 5 tokens/s on a 13-year-old Xeon without a GPU").
// NVFP4: E2M1 codes, one E4M3 scale per 16 consecutive values, one fp32 scale per tensor;
// the down matrix stored neuron-contiguous ("Running NVIDIA's new 120B Nemotron-3.5-Super
// on an 8GB GPU", "How the engine works", steps 1 and 4).
//
// Every decision that turns a float into a code is taken in fp32 with IEEE round-to-
// nearest operations written out (__fdiv_rn, __fmul_rn, __frcp_rn) and the hardware
// conversions cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32, so the bytes are reproducible.
#include "common.cuh"

namespace moe {

// ------------------------------------------------------------------------------- Q8_0
// One warp per block of 32 values.
__global__ void __launch_bounds__(256) q8_0_quantize_kernel(const float* __restrict__ src, int64_t n_blocks,
                                                             int64_t rows, int64_t cols, int layout,
                                                             uint8_t* __restrict__ dst) {
    const int lane = threadIdx.x & 31;
    const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (blk >= n_blocks) return;
    const int64_t nb = cols / 32;
    const int64_t b = blk % nb;
    const int64_t rr = blk / nb;            // matrix * rows + row
    const int64_t m = rr / rows;
    const int64_t r = rr % rows;

    const float x = src[rr * cols + b * 32 + lane];
    const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(x)));
    const float amax = __uint_as_float(amax_bits);
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    const int q = static_cast<int>(roundf(__fmul_rn(x, id)));
    const uint16_t dbits = __half_as_ushort(__float2half_rn(d));

    uint8_t* mat = dst + m * (rows * nb * 34);
    if (layout == MOE_LAYOUT_CANONICAL) {
        uint8_t* out = mat + (r * nb + b) * 34;
        out[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
        if (lane == 0) {
            out[0] = static_cast<uint8_t>(dbits & 0xffu);
            out[1] = static_cast<uint8_t>(dbits >> 8);
        }
    } else {
        uint8_t* panel = mat + b * rows * 34;
        panel[r * 32 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
        if (lane == 0) *reinterpret_cast<uint16_t*>(panel + rows * 32 + r * 2) = dbits;
    }
}

// ------------------------------------------------------------------------- per-channel int8
// One CTA per row: s = amax/127 and q = round-half-away(x / s), both fp32 IEEE divides (the
// per-channel int8 experts of "Squeezing a 26B MoE onto the cheapest Inferentia instance",
// section "Wall 1: the memory math"; the page gives no recipe, this is the plainest one).
// CANONICAL: codes row-major, then the fp32 row scales; DEVICE: the fp32 row scales first,
// then panels of 32 columns, each the 32 codes of every row.  grid (rows, n_mat).
__global__ void __launch_bounds__(256) int8pc_quantize_kernel(const float* __restrict__ src, int64_t rows,
                                                               int64_t cols, int layout, uint8_t* __restrict__ dst) {
    const int64_t r = blockIdx.x, m = blockIdx.y;
    const float* x = src + (m * rows + r) * cols;
    uint32_t mx = 0;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) mx = max(mx, __float_as_uint(fabsf(x[c])));
    mx = __reduce_max_sync(0xffffffffu, mx);
    __shared__ uint32_t wmax[8];
    __shared__ float s_sc;
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) b = max(b, wmax[i]);
        s_sc = __fdiv_rn(__uint_as_float(b), 127.0f);
    }
    __syncthreads();
    const float sc = s_sc;
    uint8_t* mat = dst + m * (rows * cols + 4 * rows);
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
        const int q = sc != 0.0f ? static_cast<int>(roundf(__fdiv_rn(x[c], sc))) : 0;
        const int64_t o = layout == MOE_LAYOUT_CANONICAL ? r * cols + c : 4 * rows + (c / 32) * rows * 32 + r * 32 + c % 32;
        mat[o] = static_cast<uint8_t>(static_cast<int8_t>(q));
    }
    if (threadIdx.x == 0) {
        const uint32_t bits = __float_as_uint(sc);
        uint8_t* sp = mat + (layout == MOE_LAYOUT_CANONICAL ? rows * cols + 4 * r : 4 * r);
        for (int i = 0; i < 4; ++i) sp[i] = static_cast<uint8_t>((bits >> (8 * i)) & 0xffu);
    }
}

// --------------------------------------------------------------- Q8_0 activations (quantise-dequantise)
// The expert inputs of the activation-quantised path (the CPU engines' Q8_0 activation
// quantiser before their Q8_0 x Q8_0 block dots: "Running Gemma 4 26B at 5 tokens/s on a
// 13-year-old Xeon without a GPU", sections "A three-step fix" and "Narrowing down the cause"):
// every block of 32 along a row is coded with the weight packer's arithmetic above, and the
// kernel writes the value each code stands for, q * fp16(d), which is exact in fp32 (8 x 11
// significant bits).  The expert kernels then meet these values exactly (their f16 hi + lo
// operands carry 22 bits), so every block's code products are summed as the integers they are
// and scaled by both fp16 scales, up to fp32 rounding.  Optionally also the f16 hi / lo planes
// of the tensor-core path.  One warp per block, grid-stride.
__global__ void __launch_bounds__(256) act_q8_0_kernel(const void* __restrict__ src, int xt, int64_t n_blocks,
                                                        int64_t cols, float* __restrict__ dst,
                                                        uint16_t* __restrict__ hi, uint16_t* __restrict__ lo) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; blk < n_blocks;
         blk += warps) {
        const int64_t nb = cols / 32;
        const int64_t o = (blk / nb) * cols + (blk % nb) * 32 + lane;
        const float x = xt == MOE_F32 ? static_cast<const float*>(src)[o]
                                      : bf16_bits_to_f32(static_cast<const uint16_t*>(src)[o]);
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(x)));
        const float v = q8_0_coded_value(x, __uint_as_float(amax_bits));
        dst[o] = v;
        if (hi) {
            const __half h = __float2half_rn(v);
            hi[o] = __half_as_ushort(h);
            lo[o] = __half_as_ushort(__float2half_rn(v - __half2float(h)));
        }
    }
}

// ------------------------------------------------------------------------------- NVFP4
// Per-matrix amax as uint bits (non-negative floats order like their bit patterns).
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const float* __restrict__ src, int64_t per_mat,
                                                          uint32_t* __restrict__ amax_bits) {
    const int64_t m = blockIdx.y;
    const float4* p = reinterpret_cast<const float4*>(src + m * per_mat);
    const int64_t n4 = per_mat / 4;
    uint32_t mx = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 v = p[i];
        mx = max(mx, __float_as_uint(fabsf(v.x)));
        mx = max(mx, __float_as_uint(fabsf(v.y)));
        mx = max(mx, __float_as_uint(fabsf(v.z)));
        mx = max(mx, __float_as_uint(fabsf(v.w)));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    __shared__ uint32_t sm[8];
    if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b = max(b, sm[i]);
        atomicMax(amax_bits + m, b);
    }
}

__device__ __forceinline__ float tensor_scale_from_amax(uint32_t bits) {
    const float amax = __uint_as_float(bits);
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);   // 6 * 448
}

__global__ void nvfp4_finalize_kernel(uint32_t* amax_bits_then_scale, int64_t n_mat) {
    const int64_t m = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (m < n_mat) {
        const float st = tensor_scale_from_amax(amax_bits_then_scale[m]);
        amax_bits_then_scale[m] = __float_as_uint(st);
    }
}

__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));   // v -> low byte
    return r & 0xffu;
}

// Two values -> one byte, `lo` in bits 3:0, `hi` in bits 7:4; a zero magnitude is coded +0.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    if ((r & 0x7u) == 0) r &= 0xf0u;
    if ((r & 0x70u) == 0) r &= 0x0fu;
    return r;
}

// Quantise one block of 16 values: returns the scale byte, writes 8 code bytes.
__device__ __forceinline__ uint32_t nvfp4_block(const float* __restrict__ x16, float st, uint32_t codes[2]) {
    float v[16];
    const float4* p = reinterpret_cast<const float4*>(x16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 q = p[i];
        v[4 * i] = q.x, v[4 * i + 1] = q.y, v[4 * i + 2] = q.z, v[4 * i + 3] = q.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float six_st = __fmul_rn(6.0f, st);
    const uint32_t sb = f32_to_e4m3(__fdiv_rn(amax, six_st));
    const float dec = e4m3_to_f32(sb);
    const float denom = __fmul_rn(dec, st);
    codes[0] = codes[1] = 0;
    if (dec != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(v[2 * i], denom), __fdiv_rn(v[2 * i + 1], denom));
            codes[i / 4] |= byte << (8 * (i % 4));
        }
    }
    return sb;
}

// CANONICAL and DEVICE layouts: one thread per block of 16 values.
__global__ void __launch_bounds__(256) nvfp4_pack_kernel(const float* __restrict__ src, int64_t n_blocks,
                                                          int64_t rows, int64_t cols, int layout,
                                                          const uint32_t* __restrict__ amax_bits,
                                                          uint8_t* __restrict__ dst) {
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (blk >= n_blocks) return;
    const int64_t nb = cols / 16;
    const int64_t b = blk % nb;
    const int64_t rr = blk / nb;
    const int64_t m = rr / rows;
    const int64_t r = rr % rows;
    const float st = tensor_scale_from_amax(amax_bits[m]);
    uint32_t codes[2];
    const uint32_t sb = nvfp4_block(src + rr * cols + b * 16, st, codes);

    const int64_t mat_bytes = rows * cols / 2 + rows * cols / 16;
    uint8_t* mat = dst + m * mat_bytes;
    if (layout == MOE_LAYOUT_CANONICAL) {
        *reinterpret_cast<uint2*>(mat + r * (cols / 2) + b * 8) = make_uint2(codes[0], codes[1]);
        mat[rows * cols / 2 + r * nb + b] = static_cast<uint8_t>(sb);
    } else {   // DEVICE: panels of 64 columns
        const int64_t pnl = b / 4, sub = b % 4;
        uint8_t* panel = mat + pnl * rows * 36;
        *reinterpret_cast<uint2*>(panel + r * 32 + sub * 8) = make_uint2(codes[0], codes[1]);
        panel[rows * 32 + r * 4 + sub] = static_cast<uint8_t>(sb);
    }
}

// NEURON layout (down matrices [rows = d][cols = f]): one thread per (row pair, group of
// 16 neurons), so that each output byte (rows 2i and 2i+1 of one neuron) has one writer.
__global__ void __launch_bounds__(256) nvfp4_pack_neuron_kernel(const float* __restrict__ src, int64_t n_items,
                                                                 int64_t rows, int64_t cols,
                                                                 const uint32_t* __restrict__ amax_bits,
                                                                 uint8_t* __restrict__ dst) {
    const int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (it >= n_items) return;
    const int64_t ng = cols / 16;
    const int64_t half_rows = rows / 2;
    const int64_t rp = it % half_rows;          // consecutive threads -> consecutive bytes
    const int64_t g = (it / half_rows) % ng;
    const int64_t m = it / (half_rows * ng);
    const float st = tensor_scale_from_amax(amax_bits[m]);
    const float* mat_src = src + m * rows * cols;
    uint32_t c0[2], c1[2];
    const uint32_t s0 = nvfp4_block(mat_src + (2 * rp) * cols + g * 16, st, c0);
    const uint32_t s1 = nvfp4_block(mat_src + (2 * rp + 1) * cols + g * 16, st, c1);

    const int64_t mat_bytes = rows * cols / 2 + rows * cols / 16;
    const int64_t rec = 16 * half_rows + rows;
    uint8_t* base = dst + m * mat_bytes + g * rec;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t lo = (c0[j / 8] >> (4 * (j % 8))) & 0xfu;   // row 2rp, neuron 16g+j
        const uint32_t hi = (c1[j / 8] >> (4 * (j % 8))) & 0xfu;   // row 2rp+1
        base[j * half_rows + rp] = static_cast<uint8_t>(lo | (hi << 4));
    }
    base[16 * half_rows + 2 * rp] = static_cast<uint8_t>(s0);
    base[16 * half_rows + 2 * rp + 1] = static_cast<uint8_t>(s1);
}

// ------------------------------------------------------------------------------- launchers
cudaError_t launch_q8_0_quantize(const float* src, int64_t n_mat, int64_t rows, int64_t cols, int layout,
                                 void* dst, cudaStream_t s) {
    const int64_t n_blocks = n_mat * rows * (cols / 32);
    const int64_t threads = n_blocks * 32;
    const int64_t grid = (threads + 255) / 256;
    q8_0_quantize_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(src, n_blocks, rows, cols, layout,
                                                                     static_cast<uint8_t*>(dst));
    return cudaGetLastError();
}

cudaError_t launch_int8pc_quantize(const float* src, int64_t n_mat, int64_t rows, int64_t cols, int layout, void* dst,
                                   cudaStream_t s) {
    int8pc_quantize_kernel<<<dim3(static_cast<unsigned>(rows), static_cast<unsigned>(n_mat)), 256, 0, s>>>(
        src, rows, cols, layout, static_cast<uint8_t*>(dst));
    return cudaGetLastError();
}

cudaError_t launch_act_q8_0(const void* src, int xt, int64_t rows, int64_t cols, float* dst, uint16_t* hi,
                            uint16_t* lo, int num_sms, cudaStream_t s) {
    const int64_t n_blocks = rows * (cols / 32);
    const int64_t want = (n_blocks * 32 + 255) / 256;
    const int64_t grid = want < 8ll * num_sms ? want : 8ll * num_sms;   // grid-stride beyond 8 CTAs per SM
    return launch_pdl(act_q8_0_kernel, dim3(static_cast<unsigned>(grid > 0 ? grid : 1)), dim3(256), 0, s, src, xt,
                      n_blocks, cols, dst, hi, lo);
}

cudaError_t launch_nvfp4_pack(const float* src, int64_t n_mat, int64_t rows, int64_t cols, int layout, void* dst,
                              float* tensor_scale, cudaStream_t s) {
    uint32_t* bits = reinterpret_cast<uint32_t*>(tensor_scale);
    cudaError_t e = cudaMemsetAsync(bits, 0, static_cast<size_t>(n_mat) * sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    const int64_t per_mat = rows * cols;
    const int64_t bx = std::min<int64_t>((per_mat / 4 + 255) / 256, 1024);
    nvfp4_amax_kernel<<<dim3(static_cast<unsigned>(bx), static_cast<unsigned>(n_mat)), 256, 0, s>>>(src, per_mat,
                                                                                                    bits);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (layout == MOE_LAYOUT_NEURON) {
        const int64_t n_items = n_mat * (rows / 2) * (cols / 16);
        nvfp4_pack_neuron_kernel<<<static_cast<unsigned>((n_items + 255) / 256), 256, 0, s>>>(
            src, n_items, rows, cols, bits, static_cast<uint8_t*>(dst));
    } else {
        const int64_t n_blocks = n_mat * rows * (cols / 16);
        nvfp4_pack_kernel<<<static_cast<unsigned>((n_blocks + 255) / 256), 256, 0, s>>>(
            src, n_blocks, rows, cols, layout, bits, static_cast<uint8_t*>(dst));
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nvfp4_finalize_kernel<<<static_cast<unsigned>((n_mat + 255) / 256), 256, 0, s>>>(bits, n_mat);
    return cudaGetLastError();
}

}  // namespace moe
