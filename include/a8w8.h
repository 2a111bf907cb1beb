/*
 * a8w8.h -- C ABI of the GB300 (sm_103a) A8W8 decode library (liba8w8.so).
 *
 * The library runs the decode hot path of a Qwen3-14B-shaped transformer with
 * INT8 weights and dynamically quantised INT8 activations on one GPU:
 * per-row activation quantisation, INT8 x INT8 -> INT32 projections with FP32
 * dequantisation, RMSNorm, per-head QK-RMSNorm + RoPE, a paged BF16 KV cache,
 * GQA decode attention, SwiGLU, and the LM head with greedy argmax; the step
 * as a replayable CUDA graph (optionally decoding on the device, greedily or
 * with sampling inside the graph); also a prefill chunk, the
 * prompt-to-first-token step, sampling beyond greedy, and two variants: the
 * INT8 KV cache with FP32 row scales and the BF16 (unquantised) layer.
 *
 * Sources, cited by page title and section:
 *   [LIB-810] "perf(qwen3-a8w8): optimize decode scheduling and data paths"
 *             (pypto-lib PR #810): "Decode scheduling", "Gate/Up INT8 path",
 *             "BF16 KV cache", "Integration note", "Validation".
 *   [SRV-48]  "Add native Qwen3 14B A8W8 serving path" (pypto-serving PR #48):
 *             loader review (per-output-channel scales), "Summary" (physical
 *             decode batch 16, startup validation), "Performance" settings.
 *   [SRV-52]  "[Feature] Add native Qwen3-14B A8W8 serving path"
 *             (pypto-serving issue #52): "Current behavior" (fused QK norm +
 *             Q RoPE), "Measurement basis" (gate/up/silu/down MLP).
 *   [SRV-61]  "Add Qwen3 A8W8 L2 runner foundation" (pypto-serving PR #61):
 *             "Summary" (block table / slot mapping packing, padded decode
 *             rows, KV page bounds validated on the host before dispatch).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller unless a
 *     parameter says "host". The library never allocates or frees device
 *     memory on these paths and never synchronises the stream, except where
 *     an entry point says so.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued asynchronously on it.
 *   - a8w8_bf16 holds a BF16 bit pattern. Matrices are row-major; weight
 *     matrices are [N, K] with K contiguous (one row per output channel).
 *   - Host-side argument validation runs before any launch; on failure
 *     nothing is enqueued and a negative a8w8_status is returned, with a
 *     message in a8w8_last_error(). Data-dependent checks (slot, block id,
 *     context length, token id, RoPE position) run on the device: the
 *     offending access is skipped and a bit is set in the device error word,
 *     read with a8w8_read_device_errors(). No kernel traps.
 *   - Pointers handed to the library must be 16-byte aligned.
 */
#ifndef A8W8_H
#define A8W8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t a8w8_bf16;

typedef enum {
    A8W8_OK = 0,
    A8W8_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad enum */
    A8W8_ERR_UNSUPPORTED_SHAPE = -2, /* shape outside what the kernels handle */
    A8W8_ERR_BOUNDS = -3,            /* an index known on the host is out of range */
    A8W8_ERR_WORKSPACE = -4,         /* workspace missing or too small */
    A8W8_ERR_CUDA = -5               /* a CUDA runtime call failed */
} a8w8_status;

/* Device error bits (a8w8_read_device_errors). */
#define A8W8_DEVERR_SLOT 0x1u        /* slot_mapping entry >= num_blocks * page */
#define A8W8_DEVERR_BLOCK 0x2u       /* block_table entry outside [0, num_blocks) */
#define A8W8_DEVERR_CTX 0x4u         /* ctx_len outside [0, max_blocks * page] */
#define A8W8_DEVERR_TOKEN 0x8u       /* token id outside [0, vocab) */
#define A8W8_DEVERR_POS 0x10u        /* RoPE position outside the table */
#define A8W8_DEVERR_TIMEOUT 0x20u    /* a bounded wait on an asynchronous copy gave up */
#define A8W8_DEVERR_ROW 0x40u        /* a8w8_prefill_step: last_rows entry outside [0, M) */

/* Message of the last failed call on this host thread ("" if none). */
const char* a8w8_last_error(void);

/* ABI version (major * 100 + minor). */
int a8w8_version(void);

/* Synchronises `stream`, then returns in *bits (host pointer) the device error
 * word of the current device accumulated since the previous read, and clears
 * it. */
a8w8_status a8w8_read_device_errors(unsigned* bits, void* stream);

/* ------------------------------------------------------------------------- */
/* Model description                                                         */
/* ------------------------------------------------------------------------- */

typedef struct {
    int hidden;           /* H (multiple of 16) */
    int num_q_heads;      /* Hq */
    int num_kv_heads;     /* Hkv, divides Hq, Hq / Hkv <= 8 */
    int head_dim;         /* D: 64 or 128 */
    int intermediate;     /* I (multiple of 16) */
    int num_layers;
    int vocab;
    int page_size;        /* tokens per KV page */
    int down_k_splits;    /* 1 or 2 (2 = the pages' two-way split-K down) */
    float rms_eps;
    int flags;            /* A8W8_FLAG_* */
} a8w8_config;

/* a8w8_config.flags: run the decode step as one persistent cooperative
 * kernel (one CTA per SM, phases separated by grid barriers) instead of one
 * kernel per operation chained with programmatic dependent launch. Applies
 * where the shape allows (batch <= 4, head_dim 128, two-way split-K down,
 * hidden and Hq*head_dim multiples of 512, intermediate a multiple of 1024);
 * otherwise the flag is ignored. Both give identical results; the separate
 * kernels are the default because they are currently faster. */
#define A8W8_FLAG_PERSISTENT_STEP 0x1

/* One layer's weights ([LIB-810] "Gate/Up INT8 path", "Integration note":
 * INT8 matrices plus FP32 per-output-channel scales; [SRV-48] loader review:
 * scales broadcast over output channels). */
typedef struct {
    const a8w8_bf16* input_norm_w;   /* [H] */
    const int8_t* w_qkv;             /* [Hq*D + 2*Hkv*D, H]: Q heads, K heads, V heads */
    const float* s_qkv;              /* [Hq*D + 2*Hkv*D] */
    const a8w8_bf16* q_norm_w;       /* [D] */
    const a8w8_bf16* k_norm_w;       /* [D] */
    const int8_t* w_o;               /* [H, Hq*D] */
    const float* s_o;                /* [H] */
    const a8w8_bf16* post_norm_w;    /* [H] */
    const int8_t* w_gate_up;         /* [2I, H]: gate rows [0, I), up rows [I, 2I) */
    const float* s_gate_up;          /* [2I] */
    const int8_t* w_down;            /* [H, I] */
    const float* s_down;             /* [H] */
} a8w8_layer_weights;

typedef struct {
    const a8w8_bf16* embed;              /* [vocab, H] */
    const a8w8_layer_weights* layers;    /* HOST array of num_layers structs */
    const a8w8_bf16* final_norm_w;       /* [H] */
    const a8w8_bf16* lm_head;            /* [vocab, H] */
} a8w8_model;

/* Optional device buffers that receive a layer's intermediates (any may be
 * NULL). They serve numerical diagnosis the way the pages' kernel
 * debug-stage switches do ([SRV-48], quoted kernel PR summary). */
typedef struct {
    a8w8_bf16* xn;                     /* [B, H] input RMSNorm output (BF16) */
    int8_t* xq;        float* xs;      /* [B, H], [B]: its quantised rows */
    a8w8_bf16* qkv;                    /* [B, Hq*D + 2*Hkv*D]: QKV projection */
    a8w8_bf16* q_rot;  a8w8_bf16* k_rot;  /* [B, Hq, D], [B, Hkv, D] after norm + RoPE */
    a8w8_bf16* attn;                   /* [B, Hq*D] attention output */
    int8_t* aq;        float* as;      /* [B, Hq*D], [B] quantised attention rows */
    a8w8_bf16* h1;                     /* [B, H] hidden after O + residual */
    a8w8_bf16* hn;                     /* [B, H] post-attention RMSNorm output */
    int8_t* hq;        float* hs;      /* [B, H], [B] its quantised rows */
    a8w8_bf16* act;                    /* [B, I] SwiGLU output */
    int8_t* actq;      float* acts;    /* [B, I], [B] quantised act rows */
} a8w8_layer_taps;

/* ------------------------------------------------------------------------- */
/* Operations                                                                */
/* ------------------------------------------------------------------------- */

/* Per-row dynamic symmetric INT8 quantisation ([LIB-810] "Decode scheduling":
 * activation quantisation batched across decode rows; "Gate/Up INT8 path":
 * quantised once per row). For each row r of x ([rows, cols] BF16, row stride
 * ldx elements): s = absmax / 127 (IEEE float32 division), q = clamp(rne(x/s),
 * -127, 127) (IEEE float32 division, ties to even); a zero row gives s = 0,
 * q = 0. Outputs q [rows, cols] int8 (dense) and row_scale [rows] float.
 * cols must be a multiple of 8 and ldx a multiple of 8 with ldx >= cols. */
a8w8_status a8w8_quant_rows(const a8w8_bf16* x, int rows, int cols, int ldx,
                            int8_t* q, float* row_scale, void* stream);

/* A8W8 projection ([LIB-810] "Gate/Up INT8 path": INT8 x INT8 -> INT32 with
 * FP32 dequantisation; "Decode scheduling": two-way K parallelism of the down
 * projection with independent partial accumulators; review "Changes": FP32
 * partials accumulated, then cast with the residual).
 *   acc_j[m][n] = sum_{k in split j} xq[m][k] * W[n][k]     (int32, exact)
 *   p_j = (float(acc_j) * x_scale[m]) * w_scale[n]            (float32)
 *   y[m][n] = bf16_rne( ((p_0 + p_1) ...) + float(residual[m][n]) )
 * xq [M, K] int8, x_scale [M], W [N, K] int8, w_scale [N], residual [M, N]
 * (nullable; may alias y), y [M, N] BF16. acc_out [M, N] int32 (nullable)
 * receives the full-K sum of the split accumulators. k_splits is 1 or 2 and
 * splits K into equal contiguous halves. 1 <= M; K a multiple of 16 with K /
 * k_splits a multiple of 16; N >= 1. */
a8w8_status a8w8_linear(const int8_t* xq, const float* x_scale, int M, int K,
                        const int8_t* W, const float* w_scale, int N, int k_splits,
                        const a8w8_bf16* residual, a8w8_bf16* y, int32_t* acc_out,
                        void* stream);

/* Fused Gate/Up projection with SwiGLU ([LIB-810] "Gate/Up INT8 path"; [SRV-52]
 * "Measurement basis"). W_gu [2I, K]: rows [0, I) gate, [I, 2I) up.
 *   g = (float(acc_gate) * x_scale[m]) * s_gu[j],  u likewise with s_gu[I + j]
 *   act[m][j] = bf16_rne( silu(g) * u ),  silu(g) = g / (1 + exp(-g)),
 * the product silu(g) * u of the float32 g and u evaluated in two-float
 * arithmetic (about 2^-44 relative) and rounded to BF16 once, so act is the
 * correctly rounded real value except within that distance of a rounding
 * boundary. acc_out [M, 2I] int32 (nullable). Shape rules as a8w8_linear. */
a8w8_status a8w8_gate_up_swiglu(const int8_t* xq, const float* x_scale, int M, int K,
                                const int8_t* W_gu, const float* s_gu, int I,
                                a8w8_bf16* act, int32_t* acc_out, void* stream);

/* The exact INT32 product of a prefill chunk's quantised rows with an INT8
 * weight matrix, on the tensor cores ([LIB-810] "Gate/Up INT8 path": INT8 x
 * INT8 -> INT32 matmuls; the step of a8w8_linear before dequantisation):
 *   acc[m][n] = sum_{k in [k0, k1)} xq[m][k] * W[n][k]     (int32, exact)
 * xq [M, K] int8, W [N, K] int8 (rows of K bytes), acc [M, N] int32 (dense).
 * K, k0 and k1 - k0 positive multiples of 64 with k1 <= K (a K split of the
 * down projection is one call per half); every pointer 16-byte aligned.
 * scratch: device memory of at least 2 * M * K bytes, owned by the caller,
 * that receives the FP16 images of xq (the tensor cores' activation operand)
 * and may be reused after the call completes on the stream.
 * Exact for codes in [-128, 127] whenever |acc| < 2^31. A bounded wait that
 * gives up sets A8W8_DEVERR_TIMEOUT in the device error word. */
a8w8_status a8w8_matmul_i8(const int8_t* xq, int M, int K, const int8_t* W, int N, int k0, int k1,
                           int32_t* acc, void* scratch, void* stream);

/* a11-a12 fused as the decode layer runs them for one or two rows: the
 * post-attention RMSNorm of x [M, K] BF16 with weight norm_w [K] BF16,
 *   xn = bf16_rne( x * 1/sqrt(mean(x^2) + eps) * norm_w ),
 * its per-row INT8 quantisation (as a8w8_quant_rows), then Gate/Up + SwiGLU
 * as a8w8_gate_up_swiglu ([LIB-810] "Gate/Up INT8 path": one activation
 * quantisation per row feeding the fused gate/up projection). The row is
 * normalised and quantised inside the projection kernel, never written out.
 * act [M, I] BF16. K a positive multiple of 16 (at most 65536); every
 * pointer 16-byte aligned. Errors as a8w8_linear. */
a8w8_status a8w8_rmsnorm_gate_up_swiglu(const a8w8_bf16* x, int M, int K,
                                        const a8w8_bf16* norm_w, float eps, const int8_t* W_gu,
                                        const float* s_gu, int I, a8w8_bf16* act, void* stream);

/* Writes k, v ([T, Hkv, D] BF16) into the paged caches at
 * slot_mapping[t] ([LIB-810] "BF16 KV cache": BF16 storage, no scale tensors;
 * [SRV-61] "Summary": slot mapping). Caches are [num_blocks * page_size, Hkv,
 * D] BF16. slot < 0 skips the token (padded row); slot >= num_blocks *
 * page_size is skipped and flags A8W8_DEVERR_SLOT. */
a8w8_status paged_kv_write(const a8w8_bf16* k, const a8w8_bf16* v, int T, int Hkv, int D,
                           const int32_t* slot_mapping, a8w8_bf16* k_cache,
                           a8w8_bf16* v_cache, int num_blocks, int page_size, void* stream);

/* GQA decode attention over the paged BF16 cache ([LIB-810] "BF16 KV cache":
 * attention loads BF16 K/V with no per-row dequantisation; [SRV-61]: block
 * table). For request b, query head h (KV head h / (Hq / Hkv)) and its
 * ctx_lens[b] tokens t at slot block_table[b][t / page] * page + t % page:
 *   out = sum_t softmax_t(softmax_scale * <q, K_t>) V_t
 * evaluated in two-float arithmetic (scores, exponentials and sums carried
 * as float pairs, about 2^-44 relative; split-KV partials merged with their
 * maxima) and narrowed to BF16 once, so out is the correctly rounded real
 * value except within that distance of a rounding boundary.
 * q [B, Hq, D]; block_table [B, max_blocks]; ctx_lens [B] (0 = padded row,
 * zero output); out [B, Hq, D]. ws: device workspace of at least
 * a8w8_attention_workspace_bytes(B, Hq, D, max_blocks * page_size) bytes
 * (split-KV partials; may be NULL when that is 0). D is 64 or 128, Hq / Hkv
 * <= 8. Calls that share a workspace must not overlap on the GPU. */
a8w8_status paged_decode_attention_bf16(const a8w8_bf16* q, const a8w8_bf16* k_cache,
                                        const a8w8_bf16* v_cache,
                                        const int32_t* block_table, const int32_t* ctx_lens,
                                        int B, int Hq, int Hkv, int D, int page_size,
                                        int max_blocks, int num_blocks, float softmax_scale,
                                        a8w8_bf16* out, void* ws, size_t ws_bytes,
                                        void* stream);

size_t a8w8_attention_workspace_bytes(int B, int Hq, int D, int max_ctx);

/* The same decode attention as paged_decode_attention_bf16, for callers that
 * cannot allocate device memory: a plugin whose host framework owns all GPU
 * memory and hands it no workspace, a serving loop whose memory budget is
 * fixed at start-up, or a C caller with no device allocator of its own. It
 * takes no workspace and calls no allocator (no cudaMalloc, cudaFree or
 * allocating library routine); the caller still passes q, the caches, the
 * tables and out. There is no counterpart on the source pages: this entry
 * point exists for such callers only.
 * Its split-KV partials live in one static device array built into the
 * library, A8W8_NOALLOC_SCRATCH_BYTES (8 MiB) large, held on every GPU that
 * loads the library until the process exits. A call whose partials would
 * exceed it (a8w8_attention_workspace_bytes(B, Hq, D, max_blocks * page_size)
 * > A8W8_NOALLOC_SCRATCH_BYTES) is rejected with A8W8_ERR_WORKSPACE before
 * anything is launched. The first call in each CUDA context (once per
 * device, and again after a device reset, which replaces the context) looks
 * up the array's device address with that device current, under a lock that
 * makes concurrent first calls safe; make that first call before any stream
 * capture. Every call shares the one array: calls that
 * overlap on the GPU (other streams, other host threads) race on it and must
 * be serialised by the caller. Nothing in it needs to start at zero: each call
 * writes every partial it later reads. */
#define A8W8_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
a8w8_status paged_decode_attention_bf16_noalloc(const a8w8_bf16* q, const a8w8_bf16* k_cache,
                                                const a8w8_bf16* v_cache,
                                                const int32_t* block_table,
                                                const int32_t* ctx_lens, int B, int Hq, int Hkv,
                                                int D, int page_size, int max_blocks,
                                                int num_blocks, float softmax_scale,
                                                a8w8_bf16* out, void* stream);

/* ------------------------------------------------------------------------- */
/* INT8 KV cache variant                                                     */
/* ------------------------------------------------------------------------- */

/* [LIB-810] "BF16 KV cache" names the storage that BF16 replaced: K/V cache
 * rows held as INT8 plus FP32 row scales, each token's K/V quantised when
 * written, each row dequantised where attention reads it, the scales in
 * tensors of their own. A row is one KV head's D values of one token:
 *   codes [num_blocks * page_size, Hkv, D] int8,
 *   scales [num_blocks * page_size, Hkv] float,
 * each row quantised by the activation formula of a8w8_quant_rows from its
 * BF16 values (s = absmax / 127, q = clamp(rne(x / s), -127, 127)), and read
 * back as code * s. D is 64 or 128. */

/* Quantises k, v ([T, Hkv, D] BF16) row by row into the INT8 cache at
 * slot_mapping[t]. slot < 0 skips the token; slot >= num_blocks * page_size
 * is skipped and flags A8W8_DEVERR_SLOT. */
a8w8_status paged_kv_write_i8(const a8w8_bf16* k, const a8w8_bf16* v, int T, int Hkv, int D,
                              const int32_t* slot_mapping, int8_t* k_codes, int8_t* v_codes,
                              float* k_scale, float* v_scale, int num_blocks, int page_size,
                              void* stream);

/* paged_decode_attention_bf16 over the INT8 cache: K_t and V_t are the codes
 * times their row scales. Same arguments, workspace
 * (a8w8_attention_workspace_bytes), shape rules and errors. */
a8w8_status paged_decode_attention_i8kv(const a8w8_bf16* q, const int8_t* k_codes,
                                        const int8_t* v_codes, const float* k_scale,
                                        const float* v_scale, const int32_t* block_table,
                                        const int32_t* ctx_lens, int B, int Hq, int Hkv, int D,
                                        int page_size, int max_blocks, int num_blocks,
                                        float softmax_scale, a8w8_bf16* out, void* ws,
                                        size_t ws_bytes, void* stream);

/* a8w8_decode_layer over this layer's INT8 cache: the new token's rotated K
 * and its V are quantised per row into the cache at slot_mapping[b] (codes and
 * scale) and attention reads the dequantised rows; every other step and every
 * argument as a8w8_decode_layer (taps included; k_rot holds the BF16 rotated
 * K before quantisation). */
a8w8_status a8w8_decode_layer_i8kv(const a8w8_layer_weights* w, const a8w8_config* cfg, int B,
                                   a8w8_bf16* hidden, const int32_t* slot_mapping,
                                   const int32_t* block_table, int max_blocks, int num_blocks,
                                   const int32_t* ctx_lens, int8_t* k_codes, int8_t* v_codes,
                                   float* k_scale, float* v_scale, const float* rope, int max_pos,
                                   void* ws, size_t ws_bytes, const a8w8_layer_taps* taps,
                                   void* stream);

/* a8w8_prefill_layer over this layer's INT8 cache: every row's rotated K and
 * its V are quantised per row into the cache at its slot first, then each
 * row attends over its own ctx_lens[r] tokens (causal as a8w8_prefill_layer).
 * Arguments, shape rules and workspace as a8w8_prefill_layer. */
a8w8_status a8w8_prefill_layer_i8kv(const a8w8_layer_weights* w, const a8w8_config* cfg, int M,
                                    a8w8_bf16* hidden, const int32_t* slot_mapping,
                                    const int32_t* block_table, int max_blocks, int num_blocks,
                                    const int32_t* ctx_lens, int8_t* k_codes, int8_t* v_codes,
                                    float* k_scale, float* v_scale, const float* rope,
                                    int max_pos, void* ws, size_t ws_bytes,
                                    const a8w8_layer_taps* taps, void* stream);

/* ------------------------------------------------------------------------- */
/* BF16 (unquantised) layer variant                                          */
/* ------------------------------------------------------------------------- */

/* [LIB-810] (the kernel PR summary it quotes) and [SRV-48] "Summary" keep the
 * ordinary BF16 Qwen3-14B path beside the A8W8 one without giving its
 * arithmetic. Reading: the A8W8 layer's steps with every quantisation step
 * removed; each projection
 *   y[m][n] = bf16_rne( sum_k x[m][k] * W[n][k] (+ residual[m][n]) )
 * (products exact in float32, float32 sums), the SwiGLU epilogue
 * act = bf16_rne( silu(g) * u ) on the float32 g and u. */
typedef struct {
    const a8w8_bf16* input_norm_w;   /* [H] */
    const a8w8_bf16* w_qkv;          /* [Hq*D + 2*Hkv*D, H]: Q heads, K heads, V heads */
    const a8w8_bf16* q_norm_w;       /* [D] */
    const a8w8_bf16* k_norm_w;       /* [D] */
    const a8w8_bf16* w_o;            /* [H, Hq*D] */
    const a8w8_bf16* post_norm_w;    /* [H] */
    const a8w8_bf16* w_gate_up;      /* [2I, H]: gate rows [0, I), up rows [I, 2I) */
    const a8w8_bf16* w_down;         /* [H, I] */
} a8w8_bf16_layer_weights;

/* BF16 projection: x [M, K], W [N, K], residual [M, N] (nullable; may alias
 * y), y [M, N]. K a positive multiple of 8, at most 49152. */
a8w8_status bf16_linear(const a8w8_bf16* x, int M, int K, const a8w8_bf16* W, int N,
                        const a8w8_bf16* residual, a8w8_bf16* y, void* stream);

/* BF16 fused Gate/Up with SwiGLU: W_gu [2I, K] (gate rows, then up rows),
 * act [M, I]. Shape rules as bf16_linear. */
a8w8_status bf16_gate_up_swiglu(const a8w8_bf16* x, int M, int K, const a8w8_bf16* W_gu, int I,
                                a8w8_bf16* act, void* stream);

/* One BF16 decode layer: input RMSNorm, QKV projection, per-head QK RMSNorm,
 * RoPE, KV write, paged GQA attention (the A8W8 layer's kernels), O
 * projection + residual, post-attention RMSNorm, Gate/Up + SwiGLU, down
 * projection + residual. Arguments, caches, workspace (a8w8_workspace_bytes)
 * and errors as a8w8_decode_layer (cfg->down_k_splits is not used); taps:
 * the BF16 fields xn, qkv, q_rot, k_rot, attn, h1, hn, act. */
a8w8_status bf16_decode_layer(const a8w8_bf16_layer_weights* w, const a8w8_config* cfg, int B,
                              a8w8_bf16* hidden, const int32_t* slot_mapping,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* ctx_lens, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                              const float* rope, int max_pos, void* ws, size_t ws_bytes,
                              const a8w8_layer_taps* taps, void* stream);

/* Fills the RoPE table used by the layer ([SRV-52] "Current behavior": Q/K
 * RoPE of the fused QK-norm path; reading: Qwen3 rotate-half, theta from the
 * model). With c = cos(p * theta^(-2i/D)) and s = sin(p * theta^(-2i/D))
 * computed in double for i < D/2, p < max_pos, each split into float
 * hi + lo parts (hi = float(x), lo = float(x - hi)):
 *   rope[p][i] = c_hi, rope[p][D/2 + i] = s_hi,
 *   rope[p][D + i] = c_lo, rope[p][3D/2 + i] = s_lo.
 * rope: device [max_pos, 2 * D] float. */
a8w8_status a8w8_rope_table(float* rope, int max_pos, int D, double theta, void* stream);

/* Sampling beyond greedy, on the device ([SRV-48] "Performance": the greedy
 * step is temperature 0, top_p 1; [SRV-61] "Related": device-side sampling).
 * logits: device [B, ld] float32 (e.g. the logits output of a8w8_decode_step);
 * next_tokens: device [B] int32. Per row: temperature <= 0 gives the argmax
 * (lowest index on ties). Otherwise z = (l - max l) / temperature and
 * p = exp(z); for top_p < 1 the nucleus is {float(p) >= tau} with tau the
 * largest such value whose tokens carry at least top_p of the mass (ties at
 * tau kept); the token is the argmax over the nucleus of z_i + g_i with
 * g_i = -log(-log(u_i)), a draw from softmax(z) on the nucleus (Gumbel-max
 * rule). u_i = (floor(x / 2^8) + 1/2) / 2^24 with x the first word of
 * Philox4x32-10, key (seed low 32 bits, seed high 32 bits), counter
 * (i, row, step low 32 bits, step high 32 bits): the same (seed, step) gives
 * the same tokens. ws / ws_bytes: a8w8_sample_workspace_bytes(B, V), device
 * memory owned by the caller (its contents need no initialisation). Calls
 * that share a workspace must not overlap on the GPU. Errors: top_p outside
 * (0, 1], a non-finite temperature, ld < V, NULL pointers, a small
 * workspace. */
size_t a8w8_sample_workspace_bytes(int B, int V);
a8w8_status a8w8_sample(const float* logits, int B, int V, int ld, float temperature, float top_p,
                        uint64_t seed, uint64_t step, int32_t* next_tokens, void* ws,
                        size_t ws_bytes, void* stream);

/* Bytes of workspace a8w8_decode_layer / a8w8_decode_step need for batches of
 * up to max_B rows and block tables of max_blocks entries. */
size_t a8w8_workspace_bytes(const a8w8_config* cfg, int max_B, int max_blocks);

/* One A8W8 decode layer on B rows (the method's steps, in order): input
 * RMSNorm, per-row INT8 quantisation, QKV projection, per-head QK RMSNorm,
 * RoPE at position ctx_lens[b] - 1, KV write at slot_mapping[b], paged GQA
 * attention over ctx_lens[b] tokens (the decoded token included), quantisation,
 * O projection + residual, post-attention RMSNorm + quantisation, Gate/Up +
 * SwiGLU, quantisation, split-K down projection + residual.
 * hidden [B, H] BF16 is updated in place. k_cache / v_cache: this layer's
 * [num_blocks * page, Hkv, D] caches. slot_mapping [B], block_table
 * [B, max_blocks], ctx_lens [B]: padded rows ([SRV-61]) have slot -1 and
 * ctx_len 0; they write no KV and attend to nothing. rope: table from
 * a8w8_rope_table with max_pos rows. ws / ws_bytes: a8w8_workspace_bytes.
 * taps: NULL, or intermediates to capture. 1 <= B <= 64. */
a8w8_status a8w8_decode_layer(const a8w8_layer_weights* w, const a8w8_config* cfg, int B,
                              a8w8_bf16* hidden, const int32_t* slot_mapping,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* ctx_lens, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                              const float* rope, int max_pos, void* ws, size_t ws_bytes,
                              const a8w8_layer_taps* taps, void* stream);

/* One A8W8 prefill chunk through one layer: M token rows (of one or more
 * sequences) with the decode layer's arguments, where row r is the token at
 * position ctx_lens[r] - 1 of its sequence, whose block table row
 * block_table[r] it shares with the sequence's other rows ([SRV-52]
 * "Current behavior": the A8W8 prefill path; configuration of the pages'
 * prefill-chunk workload). Every row's rotated K and its V are written to its
 * slot first, then each row attends over its own ctx_lens[r] tokens, so the
 * chunk is causal: row r sees the cache's earlier tokens and the chunk's rows
 * of its sequence up to its own position. Results equal those of decoding the
 * rows one at a time in position order. Projections: 1-2 rows stream the
 * weights through the decode GEMV; 3-64 rows use INT8 tensor-core tiles of 16
 * rows; above 64 rows, 128 x 128 tensor-core tiles on exact FP16 images of the
 * codes with INT32 results in the workspace. 1 <= M <= 16384; attention
 * supports Hq / Hkv <= 7 and contexts of at most 64 chunks of 128 tokens
 * (A8W8_ERR_UNSUPPORTED_SHAPE otherwise). ws / ws_bytes:
 * a8w8_workspace_bytes(cfg, M, max_blocks). */
a8w8_status a8w8_prefill_layer(const a8w8_layer_weights* w, const a8w8_config* cfg, int M,
                               a8w8_bf16* hidden, const int32_t* slot_mapping,
                               const int32_t* block_table, int max_blocks, int num_blocks,
                               const int32_t* ctx_lens, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                               const float* rope, int max_pos, void* ws, size_t ws_bytes,
                               const a8w8_layer_taps* taps, void* stream);

/* One decode step: embedding gather of token_ids [B], the num_layers layers,
 * final RMSNorm, BF16 LM head with FP32 logits and greedy argmax (lowest index
 * on ties) into next_tokens [B] int32 ([SRV-48] "Performance": temperature 0,
 * top_p 1; [SRV-61] "Related": device-side embedding and sampling).
 * By default one kernel per operation, chained with programmatic dependent
 * launch: each kernel's first weight loads are in flight before it waits on
 * its predecessor. With A8W8_FLAG_PERSISTENT_STEP, where the shape allows,
 * the whole step is one persistent cooperative kernel.
 * k_caches / v_caches: HOST arrays of num_layers device cache pointers.
 * logits [B, vocab] float (nullable), final_hidden [B, H] BF16 (nullable:
 * the normalised last hidden state). Other arguments as a8w8_decode_layer. */
a8w8_status a8w8_decode_step(const a8w8_model* m, const a8w8_config* cfg, int B,
                             const int32_t* token_ids, const int32_t* slot_mapping,
                             const int32_t* block_table, int max_blocks, int num_blocks,
                             const int32_t* ctx_lens, a8w8_bf16* const* k_caches,
                             a8w8_bf16* const* v_caches, const float* rope, int max_pos,
                             int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                             void* ws, size_t ws_bytes, void* stream);

/* The prompt through the model to the first generated token: embedding
 * gather of token_ids [M], the num_layers layers as a8w8_prefill_layer (row
 * r at position ctx_lens[r] - 1 of its sequence, causal over the chunk), then
 * the final RMSNorm, BF16 LM head and greedy argmax on the S rows
 * last_rows [S] (device; each sequence's last prompt row) into
 * next_tokens [S] and, when not NULL, logits [S, vocab] float. The timed
 * quantity of a time to first token. Shape rules as a8w8_prefill_layer
 * (1 <= M <= 16384), 1 <= S <= M, intermediate or Hq*D + 2*Hkv*D at least
 * hidden; ws / ws_bytes: a8w8_workspace_bytes(cfg, M, max_blocks); caches as
 * a8w8_decode_step. */
a8w8_status a8w8_prefill_step(const a8w8_model* m, const a8w8_config* cfg, int M,
                              const int32_t* token_ids, const int32_t* slot_mapping,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* ctx_lens, a8w8_bf16* const* k_caches,
                              a8w8_bf16* const* v_caches, const float* rope, int max_pos, int S,
                              const int32_t* last_rows, int32_t* next_tokens, float* logits,
                              void* ws, size_t ws_bytes, void* stream);

/* a8w8_decode_step over INT8 caches: k_codes / v_codes / k_scales / v_scales
 * are HOST arrays of num_layers device pointers, each layer's cache laid out
 * as for a8w8_decode_layer_i8kv; every other argument as a8w8_decode_step
 * (A8W8_FLAG_PERSISTENT_STEP is ignored). */
a8w8_status a8w8_decode_step_i8kv(const a8w8_model* m, const a8w8_config* cfg, int B,
                                  const int32_t* token_ids, const int32_t* slot_mapping,
                                  const int32_t* block_table, int max_blocks, int num_blocks,
                                  const int32_t* ctx_lens, int8_t* const* k_codes,
                                  int8_t* const* v_codes, float* const* k_scales,
                                  float* const* v_scales, const float* rope, int max_pos,
                                  int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                                  void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* Replayable decode step                                                    */
/* ------------------------------------------------------------------------- */

/* A decode step captured once into a CUDA graph with programmatic dependent
 * launches between its kernels, then replayed. The graph reads its per-step
 * inputs from caller-owned device buffers given at creation -- token_ids [B],
 * slot_mapping [B], block_table [B, max_blocks], ctx_lens [B] -- and writes
 * next_tokens [B]; the caller may rewrite the inputs between replays.
 * With device_loop != 0 the graph ends with a kernel that prepares the next
 * step on the device: token_ids = next_tokens, and for every live row
 * (ctx_len > 0) the context grows by one token whose slot is taken from the
 * block table; a row whose context is full becomes a padded row (ctx_len 0,
 * slot -1). Replaying such a graph n times decodes n tokens greedily with no
 * host involvement. Creation captures on a private stream after
 * synchronising `stream`; it must not run while `stream` is being captured.
 * The model, caches, rope table, workspace, input/output buffers and optional
 * logits / final_hidden are borrowed and must outlive the graph. */
typedef struct a8w8_step_graph a8w8_step_graph;

a8w8_status a8w8_step_graph_create(a8w8_step_graph** out, const a8w8_model* m,
                                   const a8w8_config* cfg, int B, int max_blocks,
                                   int num_blocks, a8w8_bf16* const* k_caches,
                                   a8w8_bf16* const* v_caches, const float* rope,
                                   int max_pos, int32_t* token_ids, int32_t* slot_mapping,
                                   int32_t* block_table, int32_t* ctx_lens,
                                   int32_t* next_tokens, float* logits,
                                   a8w8_bf16* final_hidden, int device_loop, void* ws,
                                   size_t ws_bytes, void* stream);

/* The same replayable step with sampling beyond greedy inside the graph
 * ([SRV-61] "Related": device-side embedding and sampling; [SRV-48]
 * "Performance": temperature and top_p are sampling parameters of the
 * decode). After the LM head writes the step's logits, the graph runs the
 * sampler of a8w8_sample on them (same rule: temperature <= 0 is the argmax,
 * otherwise the Gumbel-max draw over the top_p nucleus) and writes the drawn
 * tokens to next_tokens; with device_loop they are fed back as the next
 * step's tokens. The draw of a replay uses the Philox step read from
 * step_counter (device, one uint64, 8-byte aligned, caller-owned: set it
 * before the first replay), which the graph advances by one at the end of
 * every replay, so replay n of a graph whose counter started at s draws
 * exactly what a8w8_sample(logits, ..., seed, s + n) would on that replay's
 * logits. logits (device [B, vocab] float32) is required here.
 * sample_ws / sample_ws_bytes: at least a8w8_sample_workspace_bytes(B, vocab)
 * bytes of 16-byte aligned device memory owned by the caller, used by every
 * replay (replays of graphs that share it must not overlap). The persistent
 * step form (A8W8_FLAG_PERSISTENT_STEP) is not used for a sampled graph.
 * Errors: as a8w8_step_graph_create, plus a NULL logits or step_counter, a
 * non-finite temperature, top_p outside (0, 1] and a small sampling
 * workspace. */
a8w8_status a8w8_step_graph_create_sampled(
    a8w8_step_graph** out, const a8w8_model* m, const a8w8_config* cfg, int B, int max_blocks,
    int num_blocks, a8w8_bf16* const* k_caches, a8w8_bf16* const* v_caches, const float* rope,
    int max_pos, int32_t* token_ids, int32_t* slot_mapping, int32_t* block_table,
    int32_t* ctx_lens, int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
    int device_loop, float temperature, float top_p, uint64_t seed, uint64_t* step_counter,
    void* sample_ws, size_t sample_ws_bytes, void* ws, size_t ws_bytes, void* stream);

/* Replays the step on `stream`. */
a8w8_status a8w8_step_graph_launch(a8w8_step_graph* g, void* stream);

/* End-to-end step from HOST buffers: copies token_ids [B], slot_mapping [B],
 * block_table [B, max_blocks] and ctx_lens [B] from host memory (pinned for
 * best speed) into the graph's device input buffers, replays the step, copies
 * next_tokens [B] back to host memory, and synchronises `stream`. */
a8w8_status a8w8_step_graph_run_host(a8w8_step_graph* g, const int32_t* token_ids,
                                     const int32_t* slot_mapping,
                                     const int32_t* block_table, const int32_t* ctx_lens,
                                     int32_t* next_tokens, void* stream);

void a8w8_step_graph_destroy(a8w8_step_graph* g);

#ifdef __cplusplus
}
#endif

#endif /* A8W8_H */
