// kernels.cuh -- parameter blocks and launchers of the A8W8 decode kernels.
#pragma once

#include <stddef.h>
#include <functional>
#include <stdint.h>

#include "common.cuh"

namespace a8w8 {

// Launch context: device properties and whether to chain with programmatic
// dependent launch.
struct Launch {
    cudaStream_t stream;
    int num_sms;
    bool pdl;
};

// Runs `setup` (a cudaFuncSetAttribute, a symbol lookup) once per CUDA
// context and key, under a lock: later calls in the same context return at
// once; a failed setup is retried on the next call. A device reset destroys
// the context, so the setup runs again in the new one.
cudaError_t once_per_context(const void* key, const std::function<cudaError_t()>& setup);

// ---------------------------------------------------------------------------
// Per-row quantisation
// ---------------------------------------------------------------------------
cudaError_t launch_quant_rows(const bf16* x, int rows, int cols, int ldx, int8_t* q,
                              float* s, const Launch& L);

// ---------------------------------------------------------------------------
// A8W8 GEMV (decode projections)
// ---------------------------------------------------------------------------
enum Prologue { PRO_I8 = 0, PRO_QUANT = 1, PRO_NORM_QUANT = 2 };
enum Epilogue { EPI_STORE = 0, EPI_SWIGLU = 1 };

struct GemvParams {
    const int8_t* W;        // [rows, K]; SwiGLU: rows [0, N) gate, [N, 2N) up
    const float* w_scale;   // per weight row
    int K;
    int N;                  // outputs per batch row
    int M;                  // batch rows of this launch
    // PRO_I8 input
    const int8_t* xq;       // [M, K]
    const float* x_scale;   // [M]
    // PRO_QUANT / PRO_NORM_QUANT input
    const bf16* x;          // [M, ldx]
    int ldx;
    const bf16* norm_w;     // [K] (PRO_NORM_QUANT)
    float eps;
    // epilogue
    const bf16* residual;   // [M, ldy] or null (may alias y)
    bf16* y;                // [M, ldy]
    int ldy;
    int32_t* acc_out;       // [M, N] (SwiGLU: [M, 2N]) or null
    // taps of the quantised input (written by CTA 0), may be null
    bf16* tap_x;            // [M, K] normalised BF16 row (PRO_NORM_QUANT)
    int8_t* tap_q;          // [M, K]
    float* tap_s;           // [M]
    unsigned* err;          // device error word (timeouts)
    unsigned* clear;        // CTA 0 zeroes clear[0, clear_n) after the wait (or null)
    int clear_n;
    int deep;               // streaming kernel, 1-2 rows: a ring deep enough for the
                            // CTA's whole share (up to 11 units per warp), all of it
                            // requested before the dependency wait, where it fits
    int late_ctas;          // streaming kernel: the last late_ctas CTAs take shares of
    float late_w;           // relative size late_w (0 / 1: equal shares)
};

// Largest batch tile one launch handles; bigger batches are tiled by the host.
int gemv_max_batch_tile(int K, int k_splits);
cudaError_t launch_gemv(int prologue, int epilogue, int k_splits, const GemvParams& p,
                        const Launch& L);

// Tensor-core form for batches of up to 16 rows (PRO_I8 input: p.xq and
// p.x_scale), K a multiple of 64 * k_splits; and the once-per-row
// quantisation (PRO_QUANT or PRO_NORM_QUANT of p.x, p.M rows) into xq [M, K]
// and xs [M] that feeds it (taps of p written per row).
bool gemv_mma_supported(int K, int k_splits);
cudaError_t launch_gemv_mma(int epilogue, int k_splits, const GemvParams& p, const Launch& L);
cudaError_t launch_quant_prep(int prologue, const GemvParams& p, int8_t* xq, float* xs,
                              const Launch& L);

// Prefill-sized projections (many rows): tiled tensor-core GEMM with an exact
// INT32 result in acc (gemm_acc_bytes), then the dequantisation epilogue.
// PRO_I8 input (p.xq, p.x_scale); K a multiple of 64 * k_splits.
bool gemm_supported(int K, int k_splits);
// tcgen05 form of the prefill GEMM: C[m][n] = sum_{k in [k0, k1)} X[m][k] *
// W[n][k] (INT32, exact) for the INT8 codes X [M, K] given as their FP16
// images X16 (launch_i8_to_f16), W [N, K] INT8 (rows of K bytes), into C [M,
// ldc]; k0 and k1 - k0 multiples of 64.
bool gemm_tc_supported(int K, int k_splits);
cudaError_t launch_gemm_tc(const uint16_t* X16, int M, const int8_t* W, int N, int K, int k0, int k1,
                           int32_t* C, int ldc, unsigned* err, const Launch& L);
// y[i] = the FP16 image of the code x[i] (exact), n a multiple of 16.
cudaError_t launch_i8_to_f16(const int8_t* x, size_t n, uint16_t* y, const Launch& L);
size_t gemm_acc_bytes(int M, int N, int epilogue, int k_splits);
// x16: room for the FP16 images of p.xq (p.M * p.K values).
cudaError_t launch_gemm_projection(int epilogue, int k_splits, const GemvParams& p, int32_t* acc,
                                   uint16_t* x16, const Launch& L);

// ---------------------------------------------------------------------------
// KV write and paged decode attention
// ---------------------------------------------------------------------------
cudaError_t launch_kv_write(const bf16* k, const bf16* v, int T, int Hkv, int D,
                            const int32_t* slot_mapping, bf16* k_cache, bf16* v_cache,
                            long num_slots, unsigned* err, const Launch& L);

struct AttnParams {
    // query source: q [B, q_stride] (head h at h*D), or, when fused, the QKV
    // projection rows [B, q_stride] with Q heads, then K heads, then V heads.
    const bf16* q;
    int q_stride;
    bool fused;
    const bf16* q_norm_w;   // fused: [D]
    const bf16* k_norm_w;   // fused: [D]
    const float* rope;      // fused: [max_pos, D]
    int max_pos;
    float eps;
    const int32_t* slot_mapping;  // fused: [B]
    bf16* k_cache;          // [num_blocks*page, Hkv, D]
    bf16* v_cache;
    const int32_t* block_table;   // [B, max_blocks]
    const int32_t* ctx_lens;      // [B]
    int B, Hq, Hkv, D, page, max_blocks, num_blocks;
    float scale;            // softmax scale as a float pair scale + scale_lo
    float scale_lo;
    bf16* out;              // [B, Hq*D]
    float* part;            // split partials, [B, Hq, splits, 2 D + 4]
    unsigned* tickets;      // [B, Hq] zero on entry, or null (separate combine kernel)
    unsigned* err;
    bf16* tap_q_rot;        // [B, Hq, D] or null
    bf16* tap_k_rot;        // [B, Hkv, D] or null
    bool kv_in_cache;       // every row's new K/V was written by launch_kv_prep
                            // (prefill: rows attend to each other's tokens)
};

// Tokens per attention CTA and the number of CTAs per (request, KV head).
// Token chunk per attention CTA and chunks per request. `combine_in_kernel`:
// the decode-layer form (small chunks; the last CTA of each (request, KV
// head) combines the partials, counted on AttnParams::tickets); otherwise
// the standalone form (large chunks, separate combine kernel).
int attn_chunk(int max_ctx, bool combine_in_kernel);
int attn_splits(int max_ctx, bool combine_in_kernel);
size_t attn_part_bytes(int B, int Hq, int D, int max_ctx, bool combine_in_kernel);
cudaError_t launch_attention(const AttnParams& p, const Launch& L);
// Grouped form for large batches / long contexts (decode layer only): one CTA
// per (request, KV head, 128-token chunk) for all query heads of the group.
bool attn_group_shape_ok(int Hq, int Hkv, int D, int max_ctx);
bool attn_group_supported(const AttnParams& p);
int attn_group_splits(int max_ctx);
cudaError_t launch_attn_group(const AttnParams& p, const Launch& L);
// Whether the decode-layer attention combines its split partials in the
// kernel (tickets given and contexts up to 16384 tokens).
bool in_kernel_combine(int max_ctx, bool tickets);

// INT8 KV cache variant (attn_i8.cu): codes [num_blocks*page, Hkv, D] int8 and
// row scales [num_blocks*page, Hkv] float; `a` as for the BF16 form with its
// k_cache / v_cache unused. Per-head and grouped forms.
struct AttnI8Params {
    AttnParams a;
    int8_t* k_codes;
    int8_t* v_codes;
    float* k_scale;
    float* v_scale;
};
cudaError_t launch_attention_i8(const AttnI8Params& p, const Launch& L);
// Prefill pre-pass over the INT8 cache: every row's rotated K and its V
// quantised into its slot (then launch_attention_i8 with a.kv_in_cache).
cudaError_t launch_kv_prep_i8(const AttnI8Params& p, const Launch& L);
cudaError_t launch_kv_write_i8(const bf16* k, const bf16* v, int T, int Hkv, int D,
                               const int32_t* slot_mapping, int8_t* k_codes, int8_t* v_codes,
                               float* k_scale, float* v_scale, long num_slots, unsigned* err,
                               const Launch& L);
// BF16 (unquantised) layer (gemv_bf16.cu): y[m][n] = bf16(sum_k x[m][k]
// W[n][k] (+ residual[m][n])), or with `swiglu` act[m][n] = bf16(silu(g) u)
// from the gate row n and the up row N + n of W [2N, K]. K, ldx multiples
// of 8; rows processed in tiles of bf16_gemv_batch_tile(K) (0: K too large).
struct Bf16GemvParams {
    const bf16* x;          // [M, ldx]
    int ldx;
    const bf16* W;          // [N, K] (or [2N, K] with swiglu)
    int K, N, M;
    const bf16* residual;   // [M, ldy] or null (may alias y)
    bf16* y;                // [M, ldy]
    int ldy;
};
int bf16_gemv_batch_tile(int K);
cudaError_t launch_bf16_gemv(const Bf16GemvParams& p, bool swiglu, const Launch& L);
// y[r] = bf16(x[r] / sqrt(mean(x[r]^2) + eps) * w), one CTA per row (H % 8 == 0).
cudaError_t launch_rmsnorm_rows(const bf16* x, int rows, int H, const bf16* w, float eps, bf16* y,
                                const Launch& L);

// Prefill step (gather.cu): dst[s] = src[rows[s]] ([S, H] BF16); a row index
// outside [0, n_src) gives a zero row and device error bit 0x40.
cudaError_t launch_gather_rows(const bf16* src, int H, const int32_t* rows, int S, int n_src,
                               bf16* dst, unsigned* err, const Launch& L);

// Prefill: per-head K RMSNorm + RoPE of every row's new token and the K/V
// write into the cache, before the attention (fused QKV rows in p.q).
cudaError_t launch_kv_prep(const AttnParams& p, const Launch& L);

// ---------------------------------------------------------------------------
// Embedding, RoPE table, LM head + argmax
// ---------------------------------------------------------------------------
cudaError_t launch_embed(const bf16* embed, int vocab, int H, const int32_t* token_ids, int B,
                         bf16* hidden, unsigned long long* argmax_keys, unsigned* argmax_ticket,
                         unsigned* err, const Launch& L);

cudaError_t launch_rope_table(float* rope, int max_pos, int D, double theta, cudaStream_t s);

// Sampling beyond greedy (sample.cu): temperature and top-p by the Gumbel-max
// rule with Philox4x32-10 noise; ws [B][V][2] floats when 0 < top_p < 1. With
// step_ptr the step is read on the device and advanced by one after the
// token is picked (the form a captured step graph replays).
size_t sample_workspace_bytes(int B, int V);
cudaError_t launch_sample(const float* logits, int B, int V, int ld, float T, float top_p,
                          uint64_t seed, uint64_t step, float* ws, int32_t* out, const Launch& L,
                          uint64_t* step_ptr = nullptr);

struct LmHeadParams {
    const bf16* hidden;     // [M, H] (pre final norm)
    const bf16* norm_w;     // [H]
    float eps;
    const bf16* W;          // [V, H]
    int H, V, M;
    float* logits;          // [M, V] or null
    bf16* final_hidden;     // [M, H] or null
    unsigned long long* keys;   // [M] argmax keys (zero on entry)
    unsigned* ticket;       // zero on entry
    int32_t* next_tokens;   // [M]
};
int lmhead_max_batch_tile();

// Device-side decode loop: next step's token ids from this step's argmax, the
// context advanced by one position with its slot from the block table.
cudaError_t launch_advance(int32_t* token_ids, int32_t* slot_mapping, const int32_t* block_table,
                           int32_t* ctx_lens, const int32_t* next_tokens, int B, int max_blocks,
                           int page, const Launch& L);
cudaError_t launch_lmhead_argmax(const LmHeadParams& p, const Launch& L);

// ---------------------------------------------------------------------------
// Persistent decode step (one cooperative launch per step, batch <= 4)
// ---------------------------------------------------------------------------
constexpr int kMaxStepLayers = 64;

struct StepLayer {
    const bf16* input_norm_w;
    const int8_t* w_qkv;
    const float* s_qkv;
    const bf16* q_norm_w;
    const bf16* k_norm_w;
    const int8_t* w_o;
    const float* s_o;
    const bf16* post_norm_w;
    const int8_t* w_gate_up;
    const float* s_gate_up;
    const int8_t* w_down;
    const float* s_down;
};

struct StepParams {
    int B, H, Hq, Hkv, D, I, vocab, page, max_blocks, num_blocks, max_pos, L, down_splits;
    int device_loop;
    float eps;
    float attn_scale, attn_scale_lo;   // 1 / sqrt(D) as a float pair
    const bf16* embed;
    const bf16* final_norm_w;
    const bf16* lm_head;
    const float* rope;
    int32_t* token_ids;
    int32_t* slot_mapping;
    int32_t* block_table;
    int32_t* ctx_lens;
    int32_t* next_tokens;
    float* logits;
    bf16* final_hidden;
    bf16* hidden;
    bf16* qkv;
    bf16* attn;
    bf16* act;
    float* part;
    unsigned long long* keys;
    unsigned* ticket;
    unsigned* bar;          // [0] arrivals, [1] abort flag; zero at launch
    unsigned* err;
    StepLayer layers[kMaxStepLayers];
    bf16* k_cache[kMaxStepLayers];
    bf16* v_cache[kMaxStepLayers];
};

// Whether the persistent step kernel can run this shape on the current device.
bool step_supported(int B, int D, int L, int H, int I, int Hq, int Hkv, int max_ctx, int num_sms);
cudaError_t launch_step(const StepParams& p, const Launch& L);

}  // namespace a8w8
