/*
 * qgemv.h -- C ABI of the GB300 (sm_103a) quantized GEMV / skinny GEMM library
 * (libqgemv.so).
 *
 * What it computes (sources are web pages; cited by title and section):
 *
 *  qgemv_w4a16 / qgemm_w4a16_skinny
 *    "MLX Runner: An Inference Engine You Can Read", section "Architecture:
 *    one command buffer per token": each group of weights is stored as 4-bit
 *    integer codes plus one scale and one bias, weight = scale x code + bias,
 *    and the decode kernels multiply against the packed codes directly without
 *    ever storing a dequantized copy. Section "Optimized against a known
 *    ceiling": decode reads nearly every weight once, so it is bounded by
 *    memory bandwidth. The skinny form (several activation rows sharing one
 *    weight read) is the continuous batcher of "Krill Teardown", section
 *    "Core mechanisms", and the 16-token tree verification of the Uzu article,
 *    section "Producing several tokens from one model pass".
 *
 *  moe_mxfp4_expert_forward
 *    "Running Kimi K3 (2.8T) on one Apple Silicon Mac" (Deltafin), section
 *    "How it works": the router selects 16 experts per token and only those
 *    experts' weights are read; section "Technical approach / compute": the
 *    expert GEMV decodes MXFP4 (E2M1 codes, E8M0 block scale applied to the
 *    fp32 exponent) in the same pass as the multiply.
 *
 *  hadamard32_quant_i8 / gemm_w8a8_i32
 *    Uzu article, section "How Uzu optimizes bytes and tokens per pass":
 *    activations are quantized to 8 bits at run time so both matmul operands
 *    are integers; before quantization a block-diagonal randomized Hadamard
 *    transform (random sign flips, then a +-1 Hadamard per 32-value block)
 *    spreads outliers, and it is exactly invertible.
 *
 * Conventions shared by every entry point
 *  - Every array pointer is a DEVICE pointer (global memory of the current
 *    device). The caller allocates and owns all of them; the library never
 *    allocates device memory and keeps no per-call state.
 *  - Arrays are dense, row-major, contiguous. bf16 / fp16 arrays are passed as
 *    their 16-bit patterns (uint16_t). uint32_t "words" hold packed codes.
 *  - Every pointer must be 16-byte aligned (QG_ERR_MISALIGNED otherwise).
 *  - Outputs must not alias inputs.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Work is enqueued asynchronously on it; the return value reports
 *    host-side validation and launch errors only. Device-side timeouts of
 *    bounded waits are reported by qg_device_error().
 *  - Validation happens before anything is launched; on any error nothing is
 *    enqueued and the outputs are untouched.
 *  - Results are deterministic: the same inputs on the same device give
 *    bit-identical outputs (no floating-point atomics).
 *  - Accuracy: floating-point outputs y satisfy, per element,
 *        |y - y_exact| <= 2e-3 * sum_k |x_k * w_k| + 1e-5
 *    against the exact (float64) value from the same quantized inputs; the
 *    integer outputs (int8 codes, int32 products, expert indices) are exact.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QG_OK = 0,
    QG_ERR_INVALID_ARG = 1,     /* null pointer, bad size or shape           */
    QG_ERR_MISALIGNED = 2,      /* a pointer is not 16-byte aligned          */
    QG_ERR_UNSUPPORTED = 3,     /* valid request this build does not handle  */
    QG_ERR_WORKSPACE = 4,       /* workspace missing or too small            */
    QG_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed      */
    QG_ERR_DEVICE_TIMEOUT = 6   /* a kernel's bounded wait gave up           */
} qg_status;

/* Static, human-readable name of a status. Never NULL. */
QG_API const char *qg_status_string(qg_status s);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
QG_API int qg_version(void);

/*
 * qgemv_w4a16 -- y = W x for one activation row (M = 1), W stored as affine
 * 4-bit groups ("MLX Runner ...", "Architecture: one command buffer per
 * token").
 *
 *   wq         uint32 [N][K/8]: code k of row n is bits [4(k%8), 4(k%8)+3]
 *              of wq[n][k/8] (eight codes per word, lowest nibble first).
 *   scales_f16 fp16 [N][K/group_size]: scale s of (row n, group k/group_size).
 *   biases_f16 fp16 [N][K/group_size]: bias b of the same group.
 *   x_bf16     bf16 [K].
 *   y          fp32 [N] (output): y[n] = sum_k (s * q[n][k] + b) * x[k].
 *   group_size 32, 64 or 128 (other values: QG_ERR_INVALID_ARG). 64 runs on the
 *              fast kernels; 32 and 128 (the other group sizes of the affine
 *              format, "MLX Runner ...") run on the chunked kernel of
 *              qgemm_affine (one warp per row, 32-code chunks per lane; with
 *              more than 4 rows on qgemm_w4a16_skinny, one code per lane).
 *   K          multiple of group_size; N >= 1.
 *   workspace  may be NULL when ws_bytes == 0; qg_gemv_workspace_size()
 *              gives the size needed (currently 0 for every shape).
 */
QG_API qg_status qgemv_w4a16(const uint32_t *wq, const uint16_t *scales_f16,
                      const uint16_t *biases_f16, const uint16_t *x_bf16, float *y,
                      int N, int K, int group_size, void *workspace, size_t ws_bytes,
                      void *stream);

QG_API size_t qg_gemv_workspace_size(int N, int K, int group_size);

/*
 * qgemv_w4a16_group_* -- many independent M = 1 projections (each y_i = W_i x_i
 * as in qgemv_w4a16) in one persistent launch. "MLX Runner ...", section
 * "Architecture: one command buffer per token", issues all of a token's work
 * as one unit; here the row tiles of every projection in the group are streamed
 * back to back by one kernel, so the weight stream does not stop between
 * projections. The projections must not depend on each other: a launch reads
 * every x_i and writes every y_i in no particular order.
 *
 *   qg_w4_gemv_desc  one projection: the arguments of qgemv_w4a16 with the
 *                    same layouts (wq uint32 [N][K/8], scales/biases fp16
 *                    [N][K/64], x bf16 [K], y fp32 [N]); every pointer 16-byte
 *                    aligned device memory of the current device; N >= 1;
 *                    K a multiple of 2048 and at most 16384 (other K return
 *                    QG_ERR_UNSUPPORTED).
 *   qgemv_w4a16_group_create  validates the count descriptors (group_size 64;
 *                             32 and 128 return QG_ERR_UNSUPPORTED),
 *                    splits the tiles of all projections into one range per
 *                    CTA with equal bytes, and copies that plan to device
 *                    memory it allocates (cudaMalloc, synchronous copies).
 *                    The descriptors' buffers are used by every later run:
 *                    they must stay allocated until the group is destroyed.
 *                    *group is set on QG_OK.
 *   qgemv_w4a16_group_run     one launch on stream computing every y_i from
 *                    the current contents of x_i and W_i; stream-ordered, no
 *                    allocation, capturable in a CUDA graph. Run it on the
 *                    device that was current at create.
 *   qgemv_w4a16_group_destroy frees the plan (NULL is ignored); no run of the
 *                    group may be pending.
 */
typedef struct qg_w4_gemv_desc {
  const uint32_t *wq;
  const uint16_t *scales_f16;
  const uint16_t *biases_f16;
  const uint16_t *x_bf16;
  float *y;
  int N;
  int K;
} qg_w4_gemv_desc;

typedef struct qg_w4_group qg_w4_group;

QG_API qg_status qgemv_w4a16_group_create(const qg_w4_gemv_desc *descs, int count, int group_size,
                                          qg_w4_group **group);
QG_API qg_status qgemv_w4a16_group_run(const qg_w4_group *group, void *stream);
QG_API void qgemv_w4a16_group_destroy(qg_w4_group *group);

/*
 * qgemv_w4a16_chain_* -- the M = 1 projections of a decode step in dependency
 * order, as one persistent launch. "MLX Runner ...", section "Architecture:
 * one command buffer per token", issues a whole token as one unit; in a
 * decoder most projections consume the previous one's output (q, k, v -> o ->
 * gate_up -> down -> the next layer), so each projection here carries a
 * dependency level, and a projection of level L starts only after every
 * projection of the levels below L has written its y. The levels are awaited
 * inside the kernel (one counter per level in device memory) while the
 * weights keep streaming, so the weight stream does not stop between
 * dependent projections. The weights are those of qgemv_w4a16 (affine 4-bit,
 * group 64); each projection computes y = W x with x one of:
 *   QG_X_BF16    x = x_src as bf16 [K];
 *   QG_X_COPY    x[k] = bf16(x_alpha * x_src[k]), x_src fp32 [K] (an earlier
 *                level's y: the product in fp32, rounded to nearest even);
 *   QG_X_SWIGLU  x[k] = bf16(silu(g) * u * x_alpha), g = x_src[k],
 *                u = x_src[K + k], x_src fp32 [2K] (the gate/up output of a
 *                feed-forward layer), evaluated in fp32 as
 *                ((g / (1 + exp(-g))) * u) * x_alpha and rounded to nearest
 *                even.
 *
 *   qg_w4_chain_desc  one projection: wq uint32 [N][K/8], scales/biases fp16
 *                    [N][K/64] (the layouts of qgemv_w4a16), level >= 0 and
 *                    non-decreasing along the list, x_op / x_src / x_alpha as
 *                    above, y fp32 [N]; every pointer 16-byte aligned device
 *                    memory of the current device; N >= 1; K a multiple of
 *                    64 (else QG_ERR_INVALID_ARG) and at most 16384 (else
 *                    QG_ERR_UNSUPPORTED). Within one level the projections are
 *                    independent: no y may overlap another y or an x_src read
 *                    at the same level; a projection may read the y of any
 *                    lower level.
 *   qgemv_w4a16_chain_create  validates the descriptors (group_size 64; 32 and
 *                    128 return QG_ERR_UNSUPPORTED, other values
 *                    QG_ERR_INVALID_ARG), allocates device memory for a copy
 *                    of every projection's weights in the kernel's layout (the
 *                    same number of bytes as the stored weights, plus small
 *                    tables), fills it on the legacy default stream and waits
 *                    for it. The stored weights are not read afterwards (they
 *                    may be freed); x_src and y are used by every run and must
 *                    stay allocated until the chain is destroyed. *chain is
 *                    set on QG_OK.
 *   qgemv_w4a16_chain_run     one cooperative launch on stream (one CTA per
 *                    SM, all resident at once) computing every level in order
 *                    from the current x_src contents; no allocation,
 *                    capturable in a CUDA graph. Runs of one chain must not
 *                    overlap (its level counters are shared); each run leaves
 *                    them at zero, also after a device timeout. Results are
 *                    deterministic. Run it on the device current at create.
 *   qgemv_w4a16_chain_destroy frees the chain (NULL is ignored); no run may be
 *                    pending.
 *   qgemv_w4a16_chain_bytes   device bytes the chain holds.
 */
typedef enum { QG_X_BF16 = 0, QG_X_COPY = 1, QG_X_SWIGLU = 2 } qg_x_op;

typedef struct qg_w4_chain_desc {
  const uint32_t *wq;
  const uint16_t *scales_f16;
  const uint16_t *biases_f16;
  int N;
  int K;
  int level;
  int x_op;
  const void *x_src;
  float x_alpha;
  float *y;
} qg_w4_chain_desc;

typedef struct qg_w4_chain qg_w4_chain;

QG_API qg_status qgemv_w4a16_chain_create(const qg_w4_chain_desc *descs, int count, int group_size,
                                          qg_w4_chain **chain);
QG_API qg_status qgemv_w4a16_chain_run(const qg_w4_chain *chain, void *stream);
QG_API void qgemv_w4a16_chain_destroy(qg_w4_chain *chain);
QG_API size_t qgemv_w4a16_chain_bytes(const qg_w4_chain *chain);

/*
 * qgemv_w4a16_chain_trace_enable / _trace_read -- per-run timing of the chain's
 * levels (off by default). enable != 0 allocates and zeroes a buffer of
 * grid x levels x 4 uint64 (grid = qgemv_w4a16_chain_trace_shape's first
 * value, levels the number of distinct levels); enable = 0 frees it. While it
 * exists every run writes, per (CTA, level), the global timer in
 * nanoseconds when: [0] the CTA's first consumer warp reaches the level, [1]
 * its wait for the level below ends, [2] it has built the level's input, [3]
 * the CTA published its last row block of the level (0 where a CTA has no
 * work in a level; [3] keeps the latest stamp across runs until re-enabled).
 * _trace_read synchronizes the device and copies `count` values (at most the
 * buffer's) into host memory. _trace_shape writes grid and levels.
 * No run may be pending when tracing is switched.
 */
QG_API qg_status qgemv_w4a16_chain_trace_enable(qg_w4_chain *chain, int enable);
QG_API qg_status qgemv_w4a16_chain_trace_read(const qg_w4_chain *chain, uint64_t *host, size_t count);
QG_API void qgemv_w4a16_chain_trace_shape(const qg_w4_chain *chain, int *grid, int *levels);

/*
 * qgemm_w4a16_skinny -- Y = X W^T for a few activation rows, each weight read
 * once for all rows ("Krill Teardown", "Core mechanisms"; Uzu article,
 * "Producing several tokens from one model pass").
 *
 *   wq, scales_f16, biases_f16, N, K, group_size: as qgemv_w4a16.
 *   x_bf16  bf16 [M][K].
 *   y       fp32 [M][N] (output): y[m][n] = sum_k (s q[n][k] + b) x[m][k].
 *   M       1..32 (M = 1 is the same result as qgemv_w4a16).
 *   workspace / ws_bytes: at least qg_skinny_workspace_size(M, N, K,
 *           group_size) bytes of device memory, 16-byte aligned, zero-filled
 *           before its first use. Its first 1024 bytes are arrival counters
 *           that every completed call leaves at zero again; the rest is
 *           scratch (the activations' MMA operands, split-K partial sums). So
 *           one workspace serves any sequence of calls ordered on one stream;
 *           calls that may overlap need separate workspaces. After a call that
 *           reported a device error (qg_device_error) zero-fill it again.
 */
QG_API qg_status qgemm_w4a16_skinny(const uint32_t *wq, const uint16_t *scales_f16,
                             const uint16_t *biases_f16, const uint16_t *x_bf16,
                             float *y, int M, int N, int K, int group_size,
                             void *workspace, size_t ws_bytes, void *stream);

QG_API size_t qg_skinny_workspace_size(int M, int N, int K, int group_size);

/*
 * qgemm_w4a16_skinny_group_* -- many independent skinny projections (each
 * Y_i = X_i W_i^T as in qgemm_w4a16_skinny) in one persistent launch on the
 * tensor cores: the M = 16 verify batch of the Uzu article ("Producing several
 * tokens from one model pass") run over a whole list of weight matrices, the
 * row tiles of all of them streamed back to back ("MLX Runner ...",
 * "Architecture: one command buffer per token"). The projections must not
 * depend on each other: a launch reads every X_i and writes every Y_i in no
 * particular order.
 *
 *   qg_w4_gemm_desc  one projection: wq uint32 [N][K/8], scales/biases fp16
 *                    [N][K/64], x bf16 [M][K], y fp32 [M][N]; every pointer
 *                    16-byte aligned device memory of the current device;
 *                    2 <= M <= 32, N >= 1, K a multiple of 512 and at most
 *                    32768. All M of one group lie in one class, 2..16 or
 *                    17..32 (other shapes, and mixed classes, return
 *                    QG_ERR_UNSUPPORTED).
 *   qgemm_w4a16_skinny_group_create  validates the count descriptors
 *                    (group_size 64; 32 and 128 return QG_ERR_UNSUPPORTED),
 *                    encodes their TMA descriptors, splits
 *                    the row tiles of all projections into one contiguous
 *                    range per SM with equal work, and copies that plan to
 *                    device memory it allocates (cudaMalloc, synchronous
 *                    copies). The descriptors' buffers are used by every later
 *                    run: they must stay allocated until the group is
 *                    destroyed. *group is set on QG_OK.
 *   qgemm_w4a16_skinny_group_run     computes every Y_i from the current
 *                    contents of X_i and W_i: for M <= 16 two launches (the
 *                    activations' MMA operands, then the grid over all row
 *                    tiles), else one; no workspace, stream-ordered, no
 *                    allocation, capturable in a CUDA graph. Run it on the
 *                    device that was current at create.
 *   qgemm_w4a16_skinny_group_destroy frees the plan (NULL is ignored); no run
 *                    of the group may be pending.
 */
typedef struct qg_w4_gemm_desc {
  const uint32_t *wq;
  const uint16_t *scales_f16;
  const uint16_t *biases_f16;
  const uint16_t *x_bf16;
  float *y;
  int M;
  int N;
  int K;
} qg_w4_gemm_desc;

typedef struct qg_w4_skinny_group qg_w4_skinny_group;

QG_API qg_status qgemm_w4a16_skinny_group_create(const qg_w4_gemm_desc *descs, int count, int group_size,
                                                 qg_w4_skinny_group **group);
QG_API qg_status qgemm_w4a16_skinny_group_run(const qg_w4_skinny_group *group, void *stream);
QG_API void qgemm_w4a16_skinny_group_destroy(qg_w4_skinny_group *group);

/*
 * qgemm_affine -- Y = X W^T for 1..32 activation rows with affine weights at
 * any width of the format: "MLX Runner ...", "Architecture: one command buffer
 * per token" (weight = scale x code + bias at 2, 3, 4, 5, 6 or 8 bits, groups
 * of 32, 64 or 128; the codes are multiplied directly).
 *
 *   wq         uint32 [N][K*bits/32]: the codes of row n as one little-endian
 *              bit stream, code k in bits [bits*k, bits*k + bits) and bit j of
 *              the stream in bit j % 32 of word j / 32 (at 4 bits: the
 *              qgemv_w4a16 layout).
 *   bits       2, 3, 4, 5, 6 or 8.
 *   scales_f16, biases_f16  fp16 [N][K/group_size].
 *   x_bf16     bf16 [M][K]; y fp32 [M][N] (output):
 *              y[m][n] = sum_k (s * q[n][k] + b) * x[m][k].
 *   M 1..32; N >= 1; K a multiple of 32 and of group_size, at most 2^20;
 *   group_size 32, 64 or 128. Every pointer 16-byte aligned.
 * One warp per output row. Up to 4 rows: 32-code chunks per lane (at 2, 4 and
 * 8 bits codes turned into fp16 two at a time; the chunk sums of x once per
 * CTA); more rows: one code per lane (correct, not tuned). 4-bit g64
 * projections have the fast entry points above. Results are deterministic.
 * Errors: QG_ERR_INVALID_ARG, QG_ERR_MISALIGNED.
 */
QG_API qg_status qgemm_affine(const uint32_t *wq, int bits, const uint16_t *scales_f16,
                              const uint16_t *biases_f16, const uint16_t *x_bf16, float *y, int M, int N,
                              int K, int group_size, void *stream);

/*
 * qgemv_w8a16 -- y = W x for one activation row with row-int8 weights: the
 * packed int8 output head of "Running Kimi K3 (2.8T) on one Apple Silicon Mac"
 * (Deltafin), "Technical approach / compute" (the row-int8 checkpoint used
 * directly by a weight-only quantized matmul).
 *
 *   wq         int8 [N][K], row-major, 16-byte aligned; any int8 code.
 *   scales     fp32 [N]: scale s[n] of row n.
 *   x_bf16     bf16 [K], 16-byte aligned.
 *   y          fp32 [N] (output): y[n] = s[n] * sum_k q[n][k] * x[k].
 *   K          multiple of 16, at most 65536; N >= 1.
 *   Float results meet |y - y_ref| <= 2e-3 * sum_k |s q x| + 1e-5 against an
 *   exact evaluation (products are exact; the sum is fp32).
 * Errors: QG_ERR_INVALID_ARG (null pointer, bad N or K), QG_ERR_MISALIGNED.
 */
QG_API qg_status qgemv_w8a16(const int8_t *wq, const float *scales, const uint16_t *x_bf16, float *y,
                             int N, int K, void *stream);

/*
 * moe_mxfp4_expert_forward -- routed-expert MoE layer with MXFP4 experts
 * ("Running Kimi K3 ...", "How it works" and "Technical approach / compute").
 *
 *   x_bf16         bf16 [T][H] token activations.
 *   router_logits  fp32 [T][E].
 *   gate_q, up_q   uint8 [E][I][H/2]: E2M1 codes, two per byte, element 2j in
 *                  the low nibble and 2j+1 in the high nibble.
 *   gate_e8m0, up_e8m0 uint8 [E][I][H/32]: E8M0 block scale 2^(e-127) of
 *                  each run of 32 codes along H (e = 255 is not allowed).
 *   down_q         uint8 [E][H][I/2]; down_e8m0 uint8 [E][H][I/32].
 *   T >= 1, H and I multiples of 64, 1 <= top_k <= E <= 1024, top_k <= 32.
 *   y              fp32 [T][H] (output).
 *   topk_idx       int32 [T][top_k] (output): the experts with the largest
 *                  logits, in descending logit order, ties to the lower index.
 *   topk_w         fp32 [T][top_k] (output): their softmax probabilities over
 *                  all E experts (not renormalized over the top_k).
 *   Computes, for token t and slot j with e = topk_idx[t][j], p = topk_w[t][j]:
 *       g = Wg[e] x_t, u = Wu[e] x_t, h = silu(g) * u (kept in fp32),
 *       y[t] = sum_j p * (Wd[e] h).
 *   The summation order is fixed (repeated calls give identical results) but
 *   is the kernels' own. Kernel paths: H and I multiples of 512 and T <= 32
 *   run on warp-level MMAs; 33 <= T <= 64 (T * top_k <= 1024, code arrays
 *   32-byte aligned) on block-scaled tensor-core MMAs that take the E2M1 codes
 *   and E8M0 scales as stored (activations enter as exact sums of e4m3 terms);
 *   other shapes on one warp per output row. Float outputs meet |y - y_ref| <=
 *   2e-3 * sum |p w h| + 1e-5 against an exact evaluation.
 *   Scale range: any E8M0 byte 0..254 is accepted; the warp-level MMA path
 *   reads e = 0 (2^-127) as 0, which changes a result by less than
 *   6 * 2^-127 * sum|x| per block. Weights, activations and scales must keep
 *   every product and partial sum inside the fp32 range.
 *   workspace      at least qg_moe_workspace_size(T, H, I, E, top_k) bytes,
 *                  16-byte aligned; clobbered. The fp32 activations h of pair
 *                  (t, j) are left at byte offset qg_moe_workspace_h_offset()
 *                  as an array [T*top_k][I] (row t*top_k + j), for inspection.
 */
QG_API qg_status moe_mxfp4_expert_forward(const uint16_t *x_bf16, const float *router_logits,
                                   const uint8_t *gate_q, const uint8_t *gate_e8m0,
                                   const uint8_t *up_q, const uint8_t *up_e8m0,
                                   const uint8_t *down_q, const uint8_t *down_e8m0,
                                   int T, int H, int I, int E, int top_k,
                                   float *y, int32_t *topk_idx, float *topk_w,
                                   void *workspace, size_t ws_bytes, void *stream);

QG_API size_t qg_moe_workspace_size(int T, int H, int I, int E, int top_k);
QG_API size_t qg_moe_workspace_h_offset(int T, int H, int I, int E, int top_k);

/*
 * moe_mxfp4_expert_forward_noalloc -- the same computation, arguments, layouts
 * and results as moe_mxfp4_expert_forward, for callers that cannot allocate
 * device memory when they run the layer: for example a plugin inside a host
 * inference server that is handed only its input and output buffers, a
 * runtime that reserves all device memory as one pool at start-up, or code
 * recorded while a CUDA graph is being captured (cudaMalloc is not allowed
 * during capture). The pages have no counterpart; this is a library service.
 *
 * Instead of a caller workspace it uses a scratch array of
 * QG_MOE_NOALLOC_MAX_BYTES bytes that is part of the library's device image:
 * every GPU that loads the library holds it until the process exits. The call
 * itself allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).
 *   - Problems whose workspace (qg_moe_workspace_size) exceeds
 *     QG_MOE_NOALLOC_MAX_BYTES are refused with QG_ERR_WORKSPACE before any
 *     launch; with 384 experts of 7168 x 2048 and top-16 routing that admits
 *     up to T = 32 tokens.
 *   - Device-side timeouts are reported through qg_device_error, as for the
 *     other entry points.
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents; every stage writes what it later reads, and the first
 *     kernel of each call clears the counters that must start at zero. Calls that may run at the same time on the GPU (on
 *     different streams, or from different threads without ordering) race on
 *     the array: order them on one stream.
 *   - Launches never use programmatic dependent launch (qg_set_pdl is
 *     ignored here).
 */
#define QG_MOE_NOALLOC_MAX_BYTES ((size_t)8 << 20)

QG_API qg_status moe_mxfp4_expert_forward_noalloc(
    const uint16_t *x_bf16, const float *router_logits, const uint8_t *gate_q,
    const uint8_t *gate_e8m0, const uint8_t *up_q, const uint8_t *up_e8m0,
    const uint8_t *down_q, const uint8_t *down_e8m0, int T, int H, int I, int E,
    int top_k, float *y, int32_t *topk_idx, float *topk_w, void *stream);

/* QG_MOE_NOALLOC_MAX_BYTES as compiled into the library. */
QG_API size_t qg_moe_noalloc_max_bytes(void);

/*
 * hadamard32_quant_i8 -- block-32 randomized Walsh-Hadamard transform and
 * per-row symmetric int8 quantization (Uzu article, "How Uzu optimizes bytes
 * and tokens per pass").
 *
 *   x_bf16     bf16 [M][K], K a multiple of 32, M >= 1; finite values (a
 *              NaN or an infinity in a row makes that row's codes and scale
 *              meaningless; nothing else is affected).
 *   sign_bits  uint32 [K/32]: bit j of word b set = negate element 32b+j
 *              before the transform. Apply the same vector to the weights.
 *   q          int8 [M][K] (output); scale fp32 [M] (output).
 *   Per row m and block b, in fp32: v_j = +-x[m][32b+j]; the butterflies with
 *   spans 1, 2, 4, 8, 16 map each pair (i, i+h) (bit h of i clear) to
 *   (a + c, a - c) (unnormalized: H H^T = 32 I). Then s_m = max|z| / 127 and
 *   q = clamp(rint(z / s_m), -127, 127) with round-half-even IEEE division;
 *   an all-zero row gives s_m = 0 and q = 0. Codes are bit-exact.
 *   Dequantization: x . w = (s_x s_w / 32) * sum_k q_x[k] q_w[k].
 */
QG_API qg_status hadamard32_quant_i8(const uint16_t *x_bf16, const uint32_t *sign_bits,
                              int8_t *q, float *scale, int M, int K, void *stream);

/*
 * gemm_w8a8_i32 -- exact integer product C[m][n] = sum_k a[m][k] * w[n][k]
 * (Uzu article, "How Uzu optimizes bytes and tokens per pass": int8 x int8 on
 * the int8 matrix path, 16 verify rows).
 *
 *   a   int8 [M][K] (activation codes, e.g. from hadamard32_quant_i8).
 *   w   int8 [N][K] (per-output-channel weight codes).
 *   c   int32 [M][N] (output), exact.
 *   1 <= M <= 32, K a multiple of 64 with K * 127 * 128 < 2^31.
 */
QG_API qg_status gemm_w8a8_i32(const int8_t *a, const int8_t *w, int32_t *c,
                        int M, int N, int K, void *stream);

/*
 * gemm_w8a8_hadamard -- the whole int8 matrix path of the Uzu article ("How
 * Uzu optimizes bytes and tokens per pass") in ONE launch: the activations'
 * block-32 randomized Hadamard transform and per-row int8 quantization, the
 * exact int8 product with the weights, and the dequantization,
 *     y[m][n] = C[m][n] * s_a[m] * s_w[n] / 32,
 * where (q_a, s_a) = hadamard32_quant_i8(x_bf16, sign_bits) bit for bit and
 * C = q_a w^T exactly (int32). The weights must carry the same transform and
 * quantizer per row (w = q_w, sw = s_w of hadamard32_quant_i8 on the weight
 * rows with the same sign_bits), so that C s_a s_w / 32 approximates x . w.
 *
 *   x_bf16     bf16 [M][K], 1 <= M <= 16; finite values (a NaN or infinity
 *              in a row makes that row's outputs meaningless).
 *   sign_bits  uint32 [K/32] as in hadamard32_quant_i8.
 *   w          int8 [N][K] (row-major), sw fp32 [N]; N >= 1.
 *   y          fp32 [M][N] (output), computed in fp32 as
 *              (float)C * s_a * (s_w * 0.03125).
 *   K          a multiple of 1024 and at most 4096 (others:
 *              QG_ERR_UNSUPPORTED; gemm_w8a8_i32 and hadamard32_quant_i8
 *              serve them).
 *   workspace / ws_bytes: at least qg_w8a8_hadamard_workspace_size(M, K)
 *              bytes of device memory, 16-byte aligned, zero-filled before
 *              its first use; every call leaves it zero-filled again, so one
 *              workspace serves any sequence of calls ordered on one stream
 *              (after a reported device timeout zero-fill it again).
 * One cooperative launch (one CTA per SM, all resident at once: the CTAs
 * share the transform and wait for each other twice); capturable in a CUDA
 * graph.
 */
QG_API qg_status gemm_w8a8_hadamard(const uint16_t *x_bf16, const uint32_t *sign_bits, const int8_t *w,
                                    const float *sw, float *y, int M, int N, int K, void *workspace,
                                    size_t ws_bytes, void *stream);
QG_API size_t qg_w8a8_hadamard_workspace_size(int M, int K);

/*
 * qg_workspace_size -- the single workspace query of the boundary: device
 * bytes the operation `op` needs for the given shape, group size 64 where
 * the operation has one (M, N, K for the W4A16 and W8A8 products; T, E,
 * top_k with N = H and K = I for the MoE; M, K for the fused Hadamard W8A8
 * product). Arguments an operation does not use are ignored. 0 for an
 * operation that needs no workspace, an unknown op or a shape the operation
 * refuses. The per-operation queries above give the same values.
 */
typedef enum {
  QG_OP_GEMV_W4A16 = 0,     /* qgemv_w4a16 */
  QG_OP_SKINNY_W4A16 = 1,   /* qgemm_w4a16_skinny */
  QG_OP_MOE_MXFP4 = 2,      /* moe_mxfp4_expert_forward */
  QG_OP_HADAMARD_I8 = 3,    /* hadamard32_quant_i8 (none) */
  QG_OP_W8A8_I32 = 4,       /* gemm_w8a8_i32 (none) */
  QG_OP_W8A8_HADAMARD = 5   /* gemm_w8a8_hadamard */
} qg_op;

QG_API size_t qg_workspace_size(int op, int M, int N, int K, int T, int E, int top_k);

/*
 * qg_set_pdl -- process-wide launch mode. With enable != 0 every kernel is
 * launched with programmatic dependent launch, so its weight streaming may
 * start while the previous kernel on the stream is still draining. Activations
 * and outputs are only touched after the dependency resolves, but WEIGHTS may
 * be read early: enable it only when no work immediately preceding a call on
 * the same stream writes that call's weight arrays. Default: off.
 */
QG_API void qg_set_pdl(int enable);

/*
 * qg_device_error -- the sticky device-side error word of the current device:
 * 0 when no kernel has given up a bounded wait, otherwise a nonzero code
 * naming where it gave up. Synchronizes the device. With clear != 0 the word
 * is reset to 0. Returns QG_ERR_DEVICE_TIMEOUT when the word was nonzero.
 */
QG_API qg_status qg_device_error(uint32_t *code, int clear);

/*
 * qg_last_cuda_error -- the CUDA runtime error code (cudaError_t value) behind
 * the most recent QG_ERR_CUDA returned to the calling thread, 0 if none has
 * been returned; qg_last_cuda_error_string gives its text. Diagnostic only.
 */
QG_API int qg_last_cuda_error(void);
QG_API const char *qg_last_cuda_error_string(void);

/*
 * qg_selftest_wait_timeout -- exercises the device-side failure reporting on
 * the current device: one small kernel on stream whose wait can never be
 * satisfied gives up after a short bound, records a code in the error word
 * and returns, so the context stays usable.
 *   kind 0  an mbarrier phase nothing arrives at, bounded by `limit` polls
 *           (1..2^22); code 0x501.
 *   kind 1  a counter in device memory nothing raises, bounded by `limit`
 *           microseconds (1..10^6); code 0x502.
 * Afterwards qg_device_error reports QG_ERR_DEVICE_TIMEOUT with that code
 * (unless an earlier code is still set: the word keeps the first). Returns
 * QG_ERR_INVALID_ARG for another kind or limit, QG_ERR_CUDA if the launch (or
 * the 4-byte counter's allocation) fails. Diagnostic only: no other entry
 * point's results depend on it.
 */
QG_API qg_status qg_selftest_wait_timeout(int kind, uint32_t limit, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
