/*
 * moe.h -- C ABI of libmoe: one routed mixture-of-experts feed-forward layer over
 * block-quantised expert weights, hand-written CUDA for sm_103a (GB300).
 *
 * The layer (x[T,d], router W[d,E], expert gate/up [E,2f,d], down [E,d,f], top-k, an
 * activation) is the one the pages keep returning to:
 *   - "Running Gemma 4 26B at 5 tokens/s on a 13-year-old Xeon without a GPU"
 *     (amuse.peoplentools.com), section "A three-step fix" / "Runtime graph fallback":
 *     per-expert gate/up matmuls over a fused [n_embd, 2*n_ff, n_experts] tensor, gate
 *     first and up second, then SiLU(gate)*up, over Q8_0 weights;
 *   - "Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU" (molayo1419.me),
 *     sections "The single most important number: bytes per token" and "How the engine
 *     works", steps 1 and 4: gateless latent experts (up 2688x1024, down 1024x2688,
 *     ReLU^2) in NVFP4, a down matrix relaid out neuron-contiguous, and a down
 *     projection that skips 16-neuron groups that are all zero; section "How we check
 *     correctness": per-(token, expert) buffers combined in a fixed order.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device memory owned by the caller; the library
 *     allocates nothing (the caller provides the workspace) and keeps no state besides
 *     per-device kernel attributes set once.
 *   - Calls are asynchronous and ordered on the given stream (NULL = legacy default).
 *   - Arguments are validated on the host before anything is launched.  On an error
 *     nothing is launched, outputs are untouched, and the status says why.  No C++
 *     exception crosses this interface.
 *   - Faults found inside a kernel (an expert index out of range in caller-supplied
 *     routing, a tensor-core wait or a grid barrier that ran past its time limit) never
 *     trap: the kernel clamps or stops, records a code in the workspace's error word, and
 *     moe_get_device_status() reports it.
 *   - Shapes: row counts and column counts must be multiples of 32 (Q8_0) or 64
 *     (NVFP4); the layer needs d a multiple of 256 and f a multiple of 32 (Q8_0) or 64
 *     (NVFP4).  Pointers must be 16-byte aligned.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t.  Declared here so that this header needs no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, k out of range, unknown enum value */
    MOE_ERR_SHAPE = 2,         /* a dimension is not a supported multiple / too large */
    MOE_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned */
    MOE_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than the size query says */
    MOE_ERR_UNSUPPORTED = 5,   /* combination not built (e.g. a layout for a format) */
    MOE_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch, attribute, copy) */
    MOE_ERR_DEVICE_CHECK = 7   /* a kernel recorded an error in the workspace (see below) */
} moe_status;

typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_RELU2 = 1 } moe_act;
/* Expert weight formats.  INT8PC: per-channel int8 (the Inferentia page, "Squeezing a 26B MoE
 * onto the cheapest Inferentia instance", section "Wall 1: the memory math": experts in int8
 * with one scale per output channel): per row s = amax/127 (fp32), q = round-half-away(x / s). */
typedef enum { MOE_W_Q8_0 = 0, MOE_W_NVFP4 = 1, MOE_W_INT8PC = 2 } moe_wfmt;
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/*
 * Byte layouts of one quantised matrix [rows, cols] (cols = the reduction dimension K).
 *
 * MOE_LAYOUT_CANONICAL
 *   Q8_0 : blocks of 32 consecutive values along a row, row-major; each block is the
 *          fp16 scale (little endian) then 32 int8 codes: 34 bytes per 32 values.
 *   NVFP4: all E2M1 codes row-major, two per byte (even element in the low nibble),
 *          then all E4M3 block scales row-major (one per 16 values).
 *   INT8PC: all int8 codes row-major, then one fp32 scale per row (little endian).
 * MOE_LAYOUT_DEVICE  (what moe_layer_forward reads for gate/up matrices, and for the
 *                     down matrix in Q8_0)
 *   Q8_0 : panel b = columns 32b..32b+31: the 32 codes of every row (rows in order),
 *          then the fp16 scale of every row.  Panel size rows*34 bytes.
 *   NVFP4: panel P = columns 64P..64P+63: the 32 code bytes of every row, then the 4
 *          scale bytes of every row.  Panel size rows*36 bytes.
 *   INT8PC: the fp32 scale of every row first, then panel b = columns 32b..32b+31: the 32
 *          codes of every row (rows in order).  Panel size rows*32 bytes.
 * MOE_LAYOUT_NEURON  (NVFP4 down matrices [d, f] only; what moe_layer_forward reads)
 *   Nemotron page, "How the engine works", step 4: for each group g of 16 neurons
 *   (columns), each neuron's codes for rows 0..rows-1 contiguous (rows/2 bytes, row r
 *   in the low nibble of byte r/2 when r is even), then the rows scale bytes of the
 *   group.  A pure byte permutation of the canonical layout, same size.
 * Every layout of a matrix has the same size (moe_q8_0_bytes / moe_nvfp4_bytes /
 * moe_int8pc_bytes); a
 * stack of n_mat matrices is the matrices back to back.
 */
typedef enum { MOE_LAYOUT_CANONICAL = 0, MOE_LAYOUT_DEVICE = 1, MOE_LAYOUT_NEURON = 2 } moe_layout;

/* Which expert kernels moe_layer_forward uses.  GEMV: weight-streaming matrix-vector
 * kernels (a few tokens per expert).  GEMM: grouped GEMMs on the tensor cores (tcgen05),
 * which need f a multiple of 64 (128 for ReLU^2) and Q8_0 or NVFP4 weights; forcing GEMM on
 * another shape or format returns MOE_ERR_UNSUPPORTED (AUTO runs INT8PC weights on the GEMV
 * kernels at every T).  AUTO takes GEMM when T*k >= 8*E and the shape allows it; for ONE
 * token with Q8_0 SwiGLU (k*f <= 16384) or NVFP4 ReLU^2 experts (d <= 8192) it runs the whole
 * layer as a single cooperative kernel, one CTA per SM, when the device supports cooperative
 * launches (the same results within the output tolerance; routing, weights and the
 * permutation bit-identical).  With supplied routing that kernel skips the router and the
 * selection; an expert repeated in idx_in takes one slot per pair, in pair order, as in the
 * other paths.  GEMV keeps the separate kernels. */
typedef enum { MOE_PATH_AUTO = 0, MOE_PATH_GEMV = 1, MOE_PATH_GEMM = 2 } moe_path;

/* How the experts see their inputs.  NONE: as given (fp32 or bf16 x; h in fp32).  Q8_0: the
 * activation-quantised path of the CPU engines ("Running Gemma 4 26B at 5 tokens/s on a
 * 13-year-old Xeon without a GPU", sections "A three-step fix" and "Narrowing down the
 * cause": Q8_0 activation quantisers feeding Q8_0 x Q8_0 block dots).  Each expert input (x
 * for gate.up; h, held in fp32, for down) is coded per block of 32 with the weight packer's
 * Q8_0 codec (see moe_quantize_act_q8_0), and every weight row meets the coded values: per
 * block, the 32 code products summed exactly, times both fp16 scales, the blocks summed in
 * fp32.  Routing still reads the unquantised x.  Q8_0 weights only. */
typedef enum { MOE_ACTQ_NONE = 0, MOE_ACTQ_Q8_0 = 1 } moe_act_quant;

/* Bytes of one quantised matrix: rows*cols/32*34 (Q8_0), rows*cols/2 + rows*cols/16
 * (NVFP4).  Returns 0 for non-positive or non-multiple sizes. */
size_t moe_q8_0_bytes(int64_t rows, int64_t cols);
size_t moe_nvfp4_bytes(int64_t rows, int64_t cols);
size_t moe_int8pc_bytes(int64_t rows, int64_t cols);   /* rows*cols + 4*rows (cols a multiple of 32) */

/*
 * moe_quantize_q8_0 -- Q8_0 weight packer (the Xeon page's Q8_0 experts; block of 32
 * int8 codes and one fp16 scale).  For every row and block of 32 along cols:
 *   d = amax/127 (fp32), id = 1/d (0 when d = 0), q = round-half-away(x*id);
 *   stored scale = fp16(d) rounded to nearest even; codes use the fp32 d.
 * src   device, fp32 [n_mat][rows][cols] row-major.
 * dst   device, n_mat * moe_q8_0_bytes(rows, cols) bytes, written in `layout`
 *       (CANONICAL or DEVICE).
 * Errors: INVALID_ARG (NULL, n_mat < 0, bad layout), SHAPE (rows or cols not a
 * positive multiple of 32), ALIGNMENT, CUDA.
 */
moe_status moe_quantize_q8_0(const float* src, int64_t n_mat, int64_t rows, int64_t cols, moe_layout layout,
                             void* dst, moe_stream_t stream);

/*
 * moe_pack_nvfp4 -- NVFP4 weight packer (Nemotron page: E2M1 values, one FP8 E4M3
 * scale per 16 consecutive values, plus one fp32 scale per tensor).  Per matrix:
 *   s_t = amax/(6*448) (1 when the matrix is all zero);
 *   per 16 along cols: sb = E4M3(amax_b/(6*s_t)), round to nearest even, saturating;
 *   per value: q = E2M1(x/(dec(sb)*s_t)), nearest even, saturating; zero codes +0.
 * src           device, fp32 [n_mat][rows][cols].
 * dst           device, n_mat * moe_nvfp4_bytes(rows, cols) bytes in `layout`
 *               (CANONICAL, DEVICE or NEURON).
 * tensor_scale  device, fp32 [n_mat]: s_t of each matrix (written).
 * Errors: INVALID_ARG, SHAPE (rows a positive multiple of 32, cols of 64), ALIGNMENT,
 * CUDA.
 */
moe_status moe_pack_nvfp4(const float* src, int64_t n_mat, int64_t rows, int64_t cols, moe_layout layout,
                          void* dst, float* tensor_scale, moe_stream_t stream);

/*
 * moe_quantize_int8pc -- per-channel int8 weight packer (MOE_W_INT8PC; Inferentia page, "Wall
 * 1: the memory math", whose page gives sizes and quality but no recipe).  Per row:
 *   s = amax/127 (fp32 IEEE divide); q = round-half-away(x / s) (fp32 IEEE divide), 0 when
 *   s = 0; codes int8, the scale stored as fp32.
 * src device fp32 [n_mat][rows][cols]; dst device n_mat * moe_int8pc_bytes(rows, cols) bytes in
 * `layout` (CANONICAL or DEVICE).
 * Errors: INVALID_ARG, SHAPE (rows and cols positive multiples of 32), ALIGNMENT, CUDA.
 */
moe_status moe_quantize_int8pc(const float* src, int64_t n_mat, int64_t rows, int64_t cols, moe_layout layout,
                               void* dst, moe_stream_t stream);

/*
 * moe_quantize_act_q8_0 -- the activation quantiser of MOE_ACTQ_Q8_0, as values: every block
 * of 32 along a row of x is coded exactly as moe_quantize_q8_0 codes weights (d = amax/127 in
 * fp32, q = round-half-away(x * (1/d)), stored scale fp16(d)) and out holds q * fp16(d), the
 * value the code stands for (exact in fp32).
 * x     device [rows][cols], fp32 or bf16 (xt).   out  device fp32 [rows][cols] (written).
 * Errors: INVALID_ARG, SHAPE (cols a positive multiple of 32), ALIGNMENT, CUDA.
 */
moe_status moe_quantize_act_q8_0(const void* x, moe_dtype xt, int64_t rows, int64_t cols, float* out,
                                 moe_stream_t stream);

/*
 * moe_router_topk -- router projection, top-k and softmax over the selected logits
 * (Inferentia page, "Wall 1": top-8 of 128 experts per token; the Nemotron page:
 * top-22 of 512).
 *   logit[t][e] = fp32 dot of x[t] and W[:, e] in one canonical order: 256 partial
 *   sums (partial l takes i = l, l+256, ... in increasing i with fused multiply-add),
 *   then a halving tree (h = 128..1: s_l += s_{l+h}).
 *   Top-k: k rounds of "largest remaining logit, lower index on ties"; slot j holds the
 *   j-th selection.  w[t][j] = exp(l_j - l_0) / sum_j' exp(l_j' - l_0), sum in slot order.
 * x         device, [T][d], fp32 or bf16 (xt).
 * W         device, fp32 [d][E] row-major.
 * idx, w    device outputs, int32 [T][k] and fp32 [T][k].
 * logits    device output, fp32 [T][E], or NULL.
 * workspace device, moe_router_workspace_bytes(T, E) bytes (may be NULL when that is 0).
 * Errors: INVALID_ARG (k < 1, k > E, k > 32, E > 1024), SHAPE (d not a multiple of
 * 256), ALIGNMENT, WORKSPACE, CUDA.
 */
size_t moe_router_workspace_bytes(int64_t T, int64_t E);
moe_status moe_router_topk(const void* x, moe_dtype xt, const float* W, int64_t T, int64_t d, int64_t E, int k,
                           int32_t* idx, float* w, float* logits, void* workspace, size_t ws_bytes,
                           moe_stream_t stream);

/* Weights and shape of one layer.  All pointers are device memory. */
typedef struct {
    int64_t d;                    /* model width (K of gate/up, rows of down) */
    int64_t f;                    /* expert width (neurons) */
    int64_t E;                    /* experts */
    int32_t k;                    /* experts per token */
    int32_t act;                  /* moe_act: SWIGLU (gate/up 2f rows) or RELU2 (up f rows) */
    int32_t wfmt;                 /* moe_wfmt */
    int32_t path;                 /* moe_path */
    const float* router_w;        /* fp32 [d][E] */
    const void* w_gate_up;        /* E matrices [rows_gu][d], MOE_LAYOUT_DEVICE, back to back;
                                     SwiGLU: rows 0..f-1 gate, f..2f-1 up */
    const void* w_down;           /* E matrices [d][f]: Q8_0 / INT8PC MOE_LAYOUT_DEVICE, NVFP4 MOE_LAYOUT_NEURON */
    const float* gate_up_tscale;  /* NVFP4: fp32 [E] tensor scales of the gate/up matrices */
    const float* down_tscale;     /* NVFP4: fp32 [E] tensor scales of the down matrices */
    const void* l2_prefetch;      /* optional, may be NULL: device bytes to pull into L2 while this
                                     layer's expert weights stream -- in a stack, the next layer's
                                     router weights, so its routing does not wait on HBM.  A hint:
                                     never read by the layer's arithmetic; 16-byte aligned */
    int64_t l2_prefetch_bytes;    /* bytes at l2_prefetch (rounded down to a multiple of 16) */
    int32_t act_quant;            /* moe_act_quant (MOE_ACTQ_Q8_0 needs Q8_0 weights) */
    int32_t flags;                /* MOE_FLAG_* bits, 0 for the default */
} moe_layer_desc;

/* Expert weight stacks in page-locked host memory, read by the GPU in place (on GB300 from the
 * Grace memory over NVLink-C2C): the GB300 form of the Nemotron page's experts kept in host RAM
 * ("Running NVIDIA's new 120B Nemotron-3.5-Super on an 8GB GPU", "How the engine works", step 4:
 * the up projection brought to the GPU, the down projection read over the bus in place, only its
 * active 16-neuron groups).  MOE_FLAG_HOST_DOWN: w_down lives in host memory (gate.up stays in
 * device memory, as the page stages it); MOE_FLAG_HOST_GATE_UP: w_gate_up too.
 * moe_layer_forward checks that each such pointer is a host allocation the device addresses at the
 * same pointer (else MOE_ERR_INVALID_ARG), runs the weight-streaming kernels (the tensor-core path,
 * which loads by TMA, returns MOE_ERR_UNSUPPORTED when forced) and issues no L2 bulk prefetch of
 * host weights.  Routing weights and tensor scales stay device memory.  Results are bitwise those
 * of the same weights in device memory on the same kernels (with many tokens per expert AUTO
 * would take the tensor-core path for device weights). */
#define MOE_FLAG_HOST_GATE_UP 1
#define MOE_FLAG_HOST_DOWN 2
#define MOE_FLAG_HOST_WEIGHTS (MOE_FLAG_HOST_GATE_UP | MOE_FLAG_HOST_DOWN)

/* Optional copies of intermediate results (device pointers, each may be NULL), and
 * optional stage-boundary events for timing: each non-NULL stage_events[i] must be a
 * cudaEvent_t created by the caller; it is recorded on the stream at boundary i:
 * 0 before routing, 1 after routing and the permutation, 2 after gate.up, 3 after the
 * down projection, 4 after the combine.  Recording works inside stream capture too. */
typedef struct {
    float* logits;     /* [T][E] fp32 (not written when routing is supplied) */
    int32_t* idx;      /* [T][k] */
    float* w;          /* [T][k] */
    int32_t* offsets;  /* [E+1]: expert e owns sorted rows offsets[e]..offsets[e+1]-1 */
    int32_t* perm;     /* [T*k]: pair id (t*k+j) at each sorted row */
    int32_t* pos;      /* [T*k]: sorted row of each pair */
    float* h;          /* [T*k][f] activations in sorted-row order (MOE_ACTQ_Q8_0: the coded values
                          the down projection read) */
    void* stage_events[5];
} moe_trace;

/* Workspace bytes moe_layer_forward needs for up to T_max tokens; 0 on a bad desc. */
size_t moe_layer_workspace_bytes(const moe_layer_desc* desc, int64_t T_max);

/*
 * moe_layer_forward -- one routed MoE layer:
 *   out[t] = sum_{j<k} w[t][j] * Expert_{idx[t][j]}(x[t]), the sum in slot order j.
 * Steps, all in this library's kernels: router + top-k + softmax (skipped when idx_in
 * is given), histogram / prefix scan / stable scatter of the T*k pairs by expert
 * (within an expert, pairs keep increasing t*k+j), grouped gate.up with the activation
 * fused (SwiGLU: SiLU(gate)*up; ReLU^2: max(z,0)^2) and a mask of 16-neuron groups
 * that hold a non-zero activation, a down projection that reads only those groups,
 * and a fixed-order combine (no atomics: bitwise deterministic run to run).
 * x          device [T][d], fp32 or bf16 (xt).
 * idx_in     device int32 [T][k] precomputed routing, or NULL; w_in device fp32 [T][k]
 *            (both or neither; each 16-byte aligned, else ALIGNMENT).  Entries outside
 *            [0, E) are clamped to a valid expert and recorded as device error 1 (see
 *            moe_get_device_status).  An expert repeated within a token's k entries is
 *            evaluated once per entry.
 * out        device fp32 [T][d] (written).
 * workspace  device, at least moe_layer_workspace_bytes(desc, T) bytes, 256-byte
 *            aligned, zero-filled before its first use (the library leaves its control
 *            words zero again after every call).
 * trace      optional copies of intermediates, or NULL.
 * T = 0 returns MOE_OK, launches nothing and touches no buffer (they may be NULL).
 * Errors: INVALID_ARG, SHAPE (d a multiple of 256 up to 65536; f a multiple of 32 (Q8_0) or
 * 64 (NVFP4) up to 32768; E a multiple of 4 up to 1024), ALIGNMENT, WORKSPACE, UNSUPPORTED, CUDA.
 */
moe_status moe_layer_forward(const moe_layer_desc* desc, const void* x, moe_dtype xt, int64_t T,
                             const int32_t* idx_in, const float* w_in, float* out, void* workspace,
                             size_t ws_bytes, const moe_trace* trace, moe_stream_t stream);

/* Number of kernels one moe_layer_forward call launches for this desc, T and routing
 * (routing_supplied != 0 when idx_in/w_in are given), for bf16 inputs on the current
 * device (1 when the one-kernel decode layer applies); -1 on a bad desc or T. */
int32_t moe_layer_forward_launches(const moe_layer_desc* desc, int64_t T, int32_t routing_supplied);

/*
 * moe_rmsnorm_bf16 -- glue between stacked layers: xo[t] = bf16(x[t] / sqrt(mean(x[t]^2)
 * + eps)), no gain; the sum of squares uses a fixed reduction order.
 * x device fp32 [T][d]; xo device bf16 bits [T][d].  Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
moe_status moe_rmsnorm_bf16(const float* x, int64_t T, int64_t d, float eps, uint16_t* xo, moe_stream_t stream);

/*
 * moe_stack_forward -- a stack of routed MoE layers for ONE token, the layers glued by the
 * RMS-norm of moe_rmsnorm_bf16:
 *   x_0 = x;  out_l = layer_l(x_l);  x_{l+1} = bf16(out_l / sqrt(mean(out_l^2) + eps)).
 * (The pages' models run their MoE layers as such a stack: Gemma-4 26B-A4B has 30, the
 * MiniMax model of "Why can super-large MoE be distributed for inference" 57.)
 * descs    n_layers layer descriptors of one shape (d, f, E, k, act, wfmt, path equal;
 *          the weights, router and L2 hint per layer).
 * x        device [1][d], fp32 or bf16 (xt): the first layer's input.
 * outs     device fp32 [n_layers][d] (written): every layer's output.
 * x_next   optional device bf16 [n_layers][d]: x_{l+1} for every l (the last one too), or NULL.
 * idx, w   optional device int32 / fp32 [n_layers][k]: each layer's routing, or both NULL.
 * workspace at least moe_layer_workspace_bytes(descs, 1) bytes, zero-filled before its first
 *          use (as for moe_layer_forward).
 * With Q8_0 or INT8PC SwiGLU layers (also with act_quant = MOE_ACTQ_Q8_0) or NVFP4 ReLU^2 or
 * SwiGLU layers, path AUTO, at most 64 layers that share act_quant and flags, and a device that
 * supports cooperative launches, the whole stack is ONE kernel launch (one CTA per SM, the
 * RMS-norm between layers inside it, bitwise equal to the layer-by-layer result); otherwise
 * each layer is a moe_layer_forward call followed by the RMS-norm.
 * Errors: those of moe_layer_forward, and SHAPE when the descriptors differ in shape.
 */
moe_status moe_stack_forward(const moe_layer_desc* descs, int32_t n_layers, const void* x, moe_dtype xt, float eps,
                             float* outs, uint16_t* x_next, int32_t* idx, float* w, void* workspace, size_t ws_bytes,
                             moe_stream_t stream);

/* Kernels one moe_stack_forward call launches (bf16 or fp32 x, current device); -1 on bad
 * descriptors. */
int32_t moe_stack_forward_launches(const moe_layer_desc* descs, int32_t n_layers, int32_t with_x_next);

/*
 * Bytes of the fixed device scratch behind moe_layer_forward_noalloc (16 MiB).
 */
#define MOE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * moe_layer_forward_noalloc -- moe_layer_forward for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call: it exists for callers that are
 * handed only input and output buffers and a stream (a plugin inside an engine that owns
 * every allocation), or that must not allocate while serving (an allocation can
 * synchronise the device, and allocation is not allowed while a stream is being
 * captured).  It computes exactly what moe_layer_forward computes, with the same
 * arguments minus the workspace and trace, and allocates nothing: its scratch is a
 * 16 MiB array inside the library (MOE_NOALLOC_SCRATCH_BYTES), which every GPU that loads
 * libmoe holds until the process exits.
 *   - The first call on a device looks up that array's device address (with the device
 *     current); make that first call before any stream capture.
 *   - Problems whose moe_layer_workspace_bytes(desc, T) exceeds the scratch are rejected
 *     with MOE_ERR_WORKSPACE (decode-sized T fits: e.g. the 512-expert, top-22 latent
 *     layer at T = 32 needs about 11 MB); use moe_layer_forward for larger T.
 *   - Every call shares the one array, so calls that may overlap on the GPU (different
 *     streams without ordering between them) race and corrupt each other's results;
 *     order them on one stream.
 *   - Each call first clears the array's control region (its device-error word and the
 *     counters the kernels use), on `stream`.  A device error of the call (1: a supplied
 *     expert index was clamped; 2: a wait ran past its limit and the output is NOT valid;
 *     3: an activation beyond the f16 range on the tensor-core path) stays in the array
 *     until the next call: read it with moe_layer_forward_noalloc_status.
 * Errors: as moe_layer_forward, plus WORKSPACE when the problem does not fit.
 */
moe_status moe_layer_forward_noalloc(const moe_layer_desc* desc, const void* x, moe_dtype xt, int64_t T,
                                     const int32_t* idx_in, const float* w_in, float* out, moe_stream_t stream);

/*
 * moe_layer_forward_noalloc_status -- moe_get_device_status for the scratch of
 * moe_layer_forward_noalloc on the current device: synchronises `stream`, reads the device
 * error word the last no-allocation call left (codes as for moe_get_device_status), clears
 * it, and returns MOE_OK or MOE_ERR_DEVICE_CHECK (the code in *device_code, may be NULL).
 * Call it on the stream of the call it reports on.  Like the entry point it allocates
 * nothing.
 */
moe_status moe_layer_forward_noalloc_status(moe_stream_t stream, int32_t* device_code);

/*
 * moe_get_device_status -- synchronises `stream`, reads the error word of a layer
 * workspace, clears it, and returns MOE_OK or MOE_ERR_DEVICE_CHECK (the device code in
 * *device_code, may be NULL):
 *   1 = an expert index outside [0, E) in supplied routing was clamped;
 *   2 = a wait passed its time limit (one second) and the kernel gave up; the output is then
 *       NOT valid.  Two waits can report it: a tensor-core (GEMM path) mbarrier wait (that
 *       kernel stops early), and a grid barrier of the one-kernel decode layer (one token,
 *       moe_layer_forward or moe_stack_forward), after which no CTA of the launch waits again
 *       and the kernel runs to its end at once (every index it reads from the workspace is
 *       clamped, so stale data cannot send an access out of its buffer);
 *   3 = the GEMM path met an activation (x or h) beyond the f16 range +-65504 that its
 *       tensor-core operands use (the output then holds inf).
 * (The draft interface's separate timeout status is folded into code 2 here.)
 */
moe_status moe_get_device_status(void* workspace, moe_stream_t stream, int32_t* device_code);

/* A static string naming a status. */
const char* moe_status_string(moe_status status);

/* Version of this interface (major*10000 + minor*100 + patch): 10300 adds act_quant to
 * moe_layer_desc, moe_quantize_act_q8_0 and moe_layer_forward_noalloc_status. */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
