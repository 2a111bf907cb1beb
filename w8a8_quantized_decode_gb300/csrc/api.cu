// api.cu -- the C ABI of liba8w8.so: argument validation, workspace layout,
// orchestration of the decode layer and step, and the replayable step graph.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "a8w8.h"
#include "kernels.cuh"

using namespace a8w8;

namespace a8w8 {
namespace {

// The id of the current CUDA context, read through the driver entry points
// (cuCtxGetCurrent, cuCtxGetId); every context gets a distinct id, so a value
// looked up in one context is stale exactly when the id differs. 0 when no
// context is current or the ids cannot be read.
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);

unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag resolved;
    std::call_once(resolved, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    void* ctx = nullptr;
    if (!get_current || get_current(&ctx) != 0 || !ctx) return 0;
    unsigned long long id = 0;
    if (!get_id || get_id(ctx, &id) != 0) return 0;
    return id;
}

std::mutex g_ctx_mutex;
// (context id, key) pairs whose setup has succeeded, and the symbol
// addresses looked up, per context id.
std::set<std::pair<unsigned long long, const void*>> g_ctx_done;
std::map<std::pair<unsigned long long, const void*>, void*> g_ctx_symbols;

}  // namespace

cudaError_t once_per_context(const void* key, const std::function<cudaError_t()>& setup) {
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_ctx_mutex);
    if (id && g_ctx_done.count({id, key})) return cudaSuccess;
    const cudaError_t e = setup();
    // the setup may have created the context: remember it under its id
    const unsigned long long after = current_context_id();
    if (e == cudaSuccess && after) g_ctx_done.insert({after, key});
    return e;
}

}  // namespace a8w8

namespace {

thread_local std::string g_last_error;

a8w8_status fail(a8w8_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
a8w8_status fail(a8w8_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

a8w8_status cuda_fail(cudaError_t e, const char* what) {
    return fail(A8W8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CUDA_TRY(expr, what)                          \
    do {                                              \
        cudaError_t e_ = (expr);                      \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

__device__ unsigned g_device_error;

// Device address of a __device__ variable in the current context, looked up
// once per context (nullptr if the lookup fails).
void* symbol_address(const void* symbol) {
    const unsigned long long id = current_context_id();
    {
        std::lock_guard<std::mutex> lock(g_ctx_mutex);
        auto it = g_ctx_symbols.find({id, symbol});
        if (id && it != g_ctx_symbols.end()) return it->second;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
    const unsigned long long after = current_context_id();
    if (after) {
        std::lock_guard<std::mutex> lock(g_ctx_mutex);
        g_ctx_symbols[{after, symbol}] = p;
    }
    return p;
}

int num_sms_current() {
    // a property of the device, not of the context
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

unsigned* device_error_word() { return static_cast<unsigned*>(symbol_address(&g_device_error)); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

Launch make_launch(void* stream, bool pdl) {
    Launch L;
    L.stream = static_cast<cudaStream_t>(stream);
    L.num_sms = num_sms_current();
    L.pdl = pdl;
    return L;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout shared by the layer and the step.
struct WsLayout {
    size_t hid, qkv, attn, act, qx, qs, gacc, x16, part, att_tk, keys, ticket, bar, total;
};

// Row counts above this use the tiled GEMM (prefill chunks).
constexpr int kGemmMinRows = 64;

WsLayout ws_layout(const a8w8_config& c, int B, int max_blocks) {
    const int D = c.head_dim;
    const size_t nqkv = (size_t)(c.num_q_heads + 2 * c.num_kv_heads) * D;
    WsLayout w;
    size_t o = 0;
    w.hid = o;
    o = round_up(o + (size_t)B * c.hidden * 2, 256);
    w.qkv = o;
    o = round_up(o + (size_t)B * nqkv * 2, 256);
    w.attn = o;
    o = round_up(o + (size_t)B * c.num_q_heads * D * 2, 256);
    w.act = o;
    o = round_up(o + (size_t)B * c.intermediate * 2, 256);
    // INT8 activation rows quantised once for the tensor-core projections
    w.qx = o;
    o = round_up(o + (size_t)B * std::max({c.hidden, c.num_q_heads * D, c.intermediate}), 256);
    w.qs = o;
    o = round_up(o + (size_t)B * 4, 256);
    // INT32 results of the tiled GEMM (prefill-sized batches only)
    w.gacc = o;
    if (B > kGemmMinRows)
        o = round_up(o + (size_t)B * std::max({nqkv, (size_t)2 * c.intermediate,
                                               (size_t)2 * c.hidden}) * 4, 256);
    // FP16 images of the INT8 activation rows, the GEMM's activation operand
    w.x16 = o;
    if (B > kGemmMinRows)
        o = round_up(o + (size_t)B * std::max({c.hidden, c.num_q_heads * D, c.intermediate}) * 2,
                     256);
    w.part = o;
    const int max_ctx = max_blocks * c.page_size;
    o = round_up(o + std::max(attn_part_bytes(B, c.num_q_heads, D, max_ctx, true),
                              attn_part_bytes(B, c.num_q_heads, D, max_ctx, false)),
                 256);
    w.att_tk = o;   // attention split tickets [B, Hq]
    o = round_up(o + (size_t)B * c.num_q_heads * 4, 256);
    w.keys = o;
    o = round_up(o + (size_t)B * 8, 256);
    w.ticket = o;
    o = round_up(o + 16, 256);
    w.bar = o;
    o = round_up(o + 16, 256);
    w.total = o;
    return w;
}

a8w8_status check_config(const a8w8_config* c) {
    if (!c) return fail(A8W8_ERR_INVALID_ARG, "config is NULL");
    if (c->hidden <= 0 || c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->intermediate <= 0 ||
        c->page_size <= 0 || c->num_layers < 0)
        return fail(A8W8_ERR_INVALID_ARG, "config sizes must be positive");
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "head_dim %d not supported (64 or 128)", c->head_dim);
    if (c->num_q_heads % c->num_kv_heads != 0 || c->num_q_heads / c->num_kv_heads > 8)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "Hq/Hkv must be an integer <= 8 (Hq=%d Hkv=%d)",
                    c->num_q_heads, c->num_kv_heads);
    if (c->hidden % 16 || c->intermediate % 16)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "hidden and intermediate must be multiples of 16");
    if (c->down_k_splits != 1 && c->down_k_splits != 2)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "down_k_splits must be 1 or 2");
    if (c->intermediate % (16 * c->down_k_splits))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "intermediate / down_k_splits must be a multiple of 16");
    if (!(c->rms_eps >= 0.0f)) return fail(A8W8_ERR_INVALID_ARG, "rms_eps must be >= 0");
    return A8W8_OK;
}

a8w8_status check_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
    for (const void* p : ptrs) {
        if (!p) return fail(A8W8_ERR_INVALID_ARG, "%s: required pointer is NULL", what);
        if (!aligned16(p)) return fail(A8W8_ERR_INVALID_ARG, "%s: pointer not 16-byte aligned", what);
    }
    return A8W8_OK;
}

a8w8_status check_layer_weights(const a8w8_layer_weights* w) {
    if (!w) return fail(A8W8_ERR_INVALID_ARG, "layer weights are NULL");
    return check_ptrs({w->input_norm_w, w->w_qkv, w->s_qkv, w->q_norm_w, w->k_norm_w, w->w_o, w->s_o,
                       w->post_norm_w, w->w_gate_up, w->s_gate_up, w->w_down, w->s_down},
                      "layer weights");
}

// Batches of at least this many rows use the tensor-core projection (their
// activation rows quantised once by a separate kernel); smaller ones the dp4a
// stream with the quantisation in each CTA's prologue.
constexpr int kMmaMinBatch = 3;

bool use_mma(int M, int K, int ks) { return M >= kMmaMinBatch && gemv_mma_supported(K, ks); }

// Runs a projection over batch tiles. `qx` / `qs` (room for M rows of K
// codes and M scales) receive the quantised rows on the tensor-core path.
cudaError_t run_gemv(int pro, int epi, int ks, GemvParams p, int M, const Launch& L,
                     int8_t* qx = nullptr, float* qs = nullptr, int32_t* gacc = nullptr,
                     uint16_t* x16 = nullptr) {
    const int Ntot = (epi == EPI_SWIGLU) ? 2 * p.N : p.N;
    if (M > kGemmMinRows && gacc && x16 && gemm_supported(p.K, ks) && (pro == PRO_I8 || (qx && qs)) &&
        !p.acc_out) {
        p.err = device_error_word();
        p.M = M;
        if (pro != PRO_I8) {
            cudaError_t e = launch_quant_prep(pro, p, qx, qs, L);
            if (e != cudaSuccess) return e;
            p.xq = qx;
            p.x_scale = qs;
        }
        return launch_gemm_projection(epi, ks, p, gacc, x16, L);
    }
    if (use_mma(M, p.K, ks) && (pro == PRO_I8 || (qx && qs))) {
        p.err = device_error_word();
        if (pro != PRO_I8) {
            GemvParams q = p;
            q.M = M;
            cudaError_t e = launch_quant_prep(pro, q, qx, qs, L);
            if (e != cudaSuccess) return e;
            p.xq = qx;
            p.x_scale = qs;
        }
        constexpr int tile = 16;
        for (int b0 = 0; b0 < M; b0 += tile) {
            GemvParams q = p;
            q.M = M - b0 < tile ? M - b0 : tile;
            q.xq = p.xq + (size_t)b0 * p.K;
            q.x_scale = p.x_scale + b0;
            if (p.residual) q.residual = p.residual + (size_t)b0 * p.ldy;
            q.y = p.y + (size_t)b0 * p.ldy;
            if (p.acc_out) q.acc_out = p.acc_out + (size_t)b0 * Ntot;
            if (b0) q.clear = nullptr;
            cudaError_t e = launch_gemv_mma(epi, ks, q, L);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    const int tile = gemv_max_batch_tile(p.K, ks);
    for (int b0 = 0; b0 < M; b0 += tile) {
        GemvParams q = p;
        q.M = M - b0 < tile ? M - b0 : tile;
        if (p.xq) q.xq = p.xq + (size_t)b0 * p.K;
        if (p.x_scale) q.x_scale = p.x_scale + b0;
        if (p.x) q.x = p.x + (size_t)b0 * p.ldx;
        if (p.residual) q.residual = p.residual + (size_t)b0 * p.ldy;
        q.y = p.y + (size_t)b0 * p.ldy;
        if (p.acc_out) q.acc_out = p.acc_out + (size_t)b0 * Ntot;
        if (p.tap_q) q.tap_q = p.tap_q + (size_t)b0 * p.K;
        if (p.tap_x) q.tap_x = p.tap_x + (size_t)b0 * p.K;
        q.err = device_error_word();
        if (p.tap_s) q.tap_s = p.tap_s + b0;
        cudaError_t e = launch_gemv(pro, epi, ks, q, L);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The INT8 KV cache of one layer: codes [slots, Hkv, D], row scales [slots, Hkv].
struct KvI8 {
    int8_t* k_codes;
    int8_t* v_codes;
    float* k_scale;
    float* v_scale;
};

// Enqueues one decode layer (no validation). With `kv8` the layer's cache is
// the INT8 one (k_cache / v_cache unused).
a8w8_status enqueue_layer(const a8w8_layer_weights* w, const a8w8_config& c, int B, bf16* hidden,
                          const int32_t* slot_mapping, const int32_t* block_table, int max_blocks,
                          int num_blocks, const int32_t* ctx_lens, bf16* k_cache, bf16* v_cache,
                          const float* rope, int max_pos, unsigned char* ws, const WsLayout& lay,
                          const a8w8_layer_taps* taps, const Launch& L, bool prefill = false,
                          const KvI8* kv8 = nullptr) {
    const int H = c.hidden, D = c.head_dim, Hq = c.num_q_heads, Hkv = c.num_kv_heads;
    const int I = c.intermediate, NQ = Hq * D, NQKV = NQ + 2 * Hkv * D;
    bf16* qkv = reinterpret_cast<bf16*>(ws + lay.qkv);
    bf16* attn = reinterpret_cast<bf16*>(ws + lay.attn);
    bf16* act = reinterpret_cast<bf16*>(ws + lay.act);
    float* part = reinterpret_cast<float*>(ws + lay.part);
    unsigned* att_tk = reinterpret_cast<unsigned*>(ws + lay.att_tk);
    int8_t* qx = reinterpret_cast<int8_t*>(ws + lay.qx);
    float* qs = reinterpret_cast<float*>(ws + lay.qs);
    int32_t* gacc = B > kGemmMinRows ? reinterpret_cast<int32_t*>(ws + lay.gacc) : nullptr;
    uint16_t* x16 = B > kGemmMinRows ? reinterpret_cast<uint16_t*>(ws + lay.x16) : nullptr;
    const a8w8_layer_taps none = {};
    const a8w8_layer_taps& T = taps ? *taps : none;

    // parameter blocks of a2-a4 (QKV), a5-a8 (attention) and a9-a10 (O)
    GemvParams g = {};
    g.W = w->w_qkv;
    g.w_scale = w->s_qkv;
    g.K = H;
    g.N = NQKV;
    g.x = reinterpret_cast<const bf16*>(hidden);
    g.ldx = H;
    g.norm_w = reinterpret_cast<const bf16*>(w->input_norm_w);
    g.eps = c.rms_eps;
    g.y = qkv;
    g.ldy = NQKV;
    g.tap_x = reinterpret_cast<bf16*>(T.xn);
    g.tap_q = T.xq;
    g.tap_s = T.xs;
    g.clear = att_tk;   // the attention that follows counts its splits there
    g.clear_n = B * Hq;
    GemvParams go = {};
    go.W = w->w_o;
    go.w_scale = w->s_o;
    go.K = NQ;
    go.N = H;
    go.x = attn;
    go.ldx = NQ;
    go.residual = hidden;
    go.y = hidden;
    go.ldy = H;
    go.tap_q = T.aq;
    go.tap_s = T.as;
    AttnParams a = {};
    a.q = qkv;
    a.q_stride = NQKV;
    a.fused = true;
    a.q_norm_w = reinterpret_cast<const bf16*>(w->q_norm_w);
    a.k_norm_w = reinterpret_cast<const bf16*>(w->k_norm_w);
    a.rope = rope;
    a.max_pos = max_pos;
    a.eps = c.rms_eps;
    a.slot_mapping = slot_mapping;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = c.page_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    {
        // 1 / sqrt(D) of the layer, as a float pair
        const double sd = 1.0 / std::sqrt((double)D);
        a.scale = (float)sd;
        a.scale_lo = (float)(sd - (double)a.scale);
    }
    a.out = attn;
    a.part = part;
    a.tickets = att_tk;
    a.err = device_error_word();
    a.tap_q_rot = reinterpret_cast<bf16*>(T.q_rot);
    a.tap_k_rot = reinterpret_cast<bf16*>(T.k_rot);

    cudaError_t e = cudaSuccess;
    {
        // a2-a4: input RMSNorm + quantisation (prologue) + QKV projection
        e = run_gemv(PRO_NORM_QUANT, EPI_STORE, 1, g, B, L, qx, qs, gacc, x16);
        if (e != cudaSuccess) return cuda_fail(e, "QKV projection");
        // a5-a8: QK norm, RoPE, KV write, paged attention
        if (kv8) {
            AttnI8Params ai = {};
            ai.a = a;
            ai.k_codes = kv8->k_codes;
            ai.v_codes = kv8->v_codes;
            ai.k_scale = kv8->k_scale;
            ai.v_scale = kv8->v_scale;
            if (prefill) {
                // every token's K/V quantised into the cache first (as below)
                e = launch_kv_prep_i8(ai, L);
                if (e != cudaSuccess) return cuda_fail(e, "prefill KV write");
                ai.a.kv_in_cache = true;
            }
            e = launch_attention_i8(ai, L);
        } else if (prefill) {
            // every token's K/V into the cache first: the chunk's rows attend to
            // each other's earlier tokens (causal by their context lengths)
            e = launch_kv_prep(a, L);
            if (e != cudaSuccess) return cuda_fail(e, "prefill KV write");
            a.kv_in_cache = true;
            e = launch_attn_group(a, L);
        } else {
            e = launch_attention(a, L);
        }
        if (e != cudaSuccess) return cuda_fail(e, "attention");
        // a9-a10: quantisation (prologue) + O projection + residual (in place);
        // the O matrix (26 MB) fits the grid's shared memory: each CTA
        // requests its whole share before waiting for the attention output
        go.deep = 1;
        // the O CTAs dispatched last land on the SMs that attention holds
        // (one CTA per query head at batch 1 and contexts up to one chunk)
        // and start after it, without their weights in shared memory: they
        // take shares of 0.8 (measured best of 0.65 / 0.8 / 1 over the
        // 40-layer step)
        if (B == 1) {
            go.late_ctas = c.num_q_heads;
            go.late_w = 0.8f;
        }
        e = run_gemv(PRO_QUANT, EPI_STORE, 1, go, B, L, qx, qs, gacc, x16);
        go.late_ctas = 0;
        if (e != cudaSuccess) return cuda_fail(e, "O projection");
    }
    if (T.qkv) {
        e = cudaMemcpyAsync(T.qkv, qkv, (size_t)B * NQKV * 2, cudaMemcpyDeviceToDevice, L.stream);
        if (e != cudaSuccess) return cuda_fail(e, "tap qkv");
    }
    if (T.attn) {
        e = cudaMemcpyAsync(T.attn, attn, (size_t)B * NQ * 2, cudaMemcpyDeviceToDevice, L.stream);
        if (e != cudaSuccess) return cuda_fail(e, "tap attn");
    }
    if (T.h1) {
        e = cudaMemcpyAsync(T.h1, hidden, (size_t)B * H * 2, cudaMemcpyDeviceToDevice, L.stream);
        if (e != cudaSuccess) return cuda_fail(e, "tap h1");
    }

    // a11-a12: post-attention RMSNorm + quantisation (prologue) + Gate/Up + SwiGLU
    g = GemvParams{};
    g.W = w->w_gate_up;
    g.w_scale = w->s_gate_up;
    g.K = H;
    g.N = I;
    g.x = hidden;
    g.ldx = H;
    g.norm_w = reinterpret_cast<const bf16*>(w->post_norm_w);
    g.eps = c.rms_eps;
    g.y = act;
    g.ldy = I;
    g.tap_x = reinterpret_cast<bf16*>(T.hn);
    g.tap_q = T.hq;
    g.tap_s = T.hs;
    e = run_gemv(PRO_NORM_QUANT, EPI_SWIGLU, 1, g, B, L, qx, qs, gacc, x16);
    if (e != cudaSuccess) return cuda_fail(e, "Gate/Up projection");
    if (T.act) {
        e = cudaMemcpyAsync(T.act, act, (size_t)B * I * 2, cudaMemcpyDeviceToDevice, L.stream);
        if (e != cudaSuccess) return cuda_fail(e, "tap act");
    }

    // a13-a14: quantisation (prologue) + split-K down projection + residual
    g = GemvParams{};
    g.W = w->w_down;
    g.w_scale = w->s_down;
    g.K = I;
    g.N = H;
    g.x = act;
    g.ldx = I;
    g.residual = hidden;
    g.y = hidden;
    g.ldy = H;
    g.tap_q = T.actq;
    g.tap_s = T.acts;
    e = run_gemv(PRO_QUANT, EPI_STORE, c.down_k_splits, g, B, L, qx, qs, gacc, x16);
    if (e != cudaSuccess) return cuda_fail(e, "down projection");
    return A8W8_OK;
}

// Enqueues one BF16 (unquantised) decode layer (no validation): the A8W8
// layer's steps without the quantisation, the same attention kernels.
a8w8_status enqueue_bf16_layer(const a8w8_bf16_layer_weights* w, const a8w8_config& c, int B,
                               bf16* hidden, const int32_t* slot_mapping,
                               const int32_t* block_table, int max_blocks, int num_blocks,
                               const int32_t* ctx_lens, bf16* k_cache, bf16* v_cache,
                               const float* rope, int max_pos, unsigned char* ws,
                               const WsLayout& lay, const a8w8_layer_taps* taps, const Launch& L) {
    const int H = c.hidden, D = c.head_dim, Hq = c.num_q_heads, Hkv = c.num_kv_heads;
    const int I = c.intermediate, NQ = Hq * D, NQKV = NQ + 2 * Hkv * D;
    bf16* xn = reinterpret_cast<bf16*>(ws + lay.hid);
    bf16* qkv = reinterpret_cast<bf16*>(ws + lay.qkv);
    bf16* attn = reinterpret_cast<bf16*>(ws + lay.attn);
    bf16* act = reinterpret_cast<bf16*>(ws + lay.act);
    unsigned* att_tk = reinterpret_cast<unsigned*>(ws + lay.att_tk);
    const a8w8_layer_taps none = {};
    const a8w8_layer_taps& T = taps ? *taps : none;
    auto tap = [&](void* dst, const void* src, size_t bytes, const char* what) -> a8w8_status {
        if (!dst) return A8W8_OK;
        cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, L.stream);
        return e == cudaSuccess ? A8W8_OK : cuda_fail(e, what);
    };
    a8w8_status st;

    // input RMSNorm, QKV projection
    cudaError_t e = launch_rmsnorm_rows(hidden, B, H, reinterpret_cast<const bf16*>(w->input_norm_w),
                                        c.rms_eps, xn, L);
    if (e != cudaSuccess) return cuda_fail(e, "input RMSNorm");
    if ((st = tap(T.xn, xn, (size_t)B * H * 2, "tap xn")) != A8W8_OK) return st;
    e = cudaMemsetAsync(att_tk, 0, (size_t)B * Hq * 4, L.stream);   // attention split tickets
    if (e != cudaSuccess) return cuda_fail(e, "clear tickets");
    Bf16GemvParams g = {};
    g.x = xn;
    g.ldx = H;
    g.W = reinterpret_cast<const bf16*>(w->w_qkv);
    g.K = H;
    g.N = NQKV;
    g.M = B;
    g.y = qkv;
    g.ldy = NQKV;
    e = launch_bf16_gemv(g, false, L);
    if (e != cudaSuccess) return cuda_fail(e, "QKV projection");
    if ((st = tap(T.qkv, qkv, (size_t)B * NQKV * 2, "tap qkv")) != A8W8_OK) return st;

    // QK norm, RoPE, KV write, paged attention: the A8W8 layer's kernels
    AttnParams a = {};
    a.q = qkv;
    a.q_stride = NQKV;
    a.fused = true;
    a.q_norm_w = reinterpret_cast<const bf16*>(w->q_norm_w);
    a.k_norm_w = reinterpret_cast<const bf16*>(w->k_norm_w);
    a.rope = rope;
    a.max_pos = max_pos;
    a.eps = c.rms_eps;
    a.slot_mapping = slot_mapping;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = c.page_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    {
        const double sd = 1.0 / std::sqrt((double)D);
        a.scale = (float)sd;
        a.scale_lo = (float)(sd - (double)a.scale);
    }
    a.out = attn;
    a.part = reinterpret_cast<float*>(ws + lay.part);
    a.tickets = att_tk;
    a.err = device_error_word();
    a.tap_q_rot = reinterpret_cast<bf16*>(T.q_rot);
    a.tap_k_rot = reinterpret_cast<bf16*>(T.k_rot);
    e = launch_attention(a, L);
    if (e != cudaSuccess) return cuda_fail(e, "attention");
    if ((st = tap(T.attn, attn, (size_t)B * NQ * 2, "tap attn")) != A8W8_OK) return st;

    // O projection + residual (in place)
    g = Bf16GemvParams{};
    g.x = attn;
    g.ldx = NQ;
    g.W = reinterpret_cast<const bf16*>(w->w_o);
    g.K = NQ;
    g.N = H;
    g.M = B;
    g.residual = hidden;
    g.y = hidden;
    g.ldy = H;
    e = launch_bf16_gemv(g, false, L);
    if (e != cudaSuccess) return cuda_fail(e, "O projection");
    if ((st = tap(T.h1, hidden, (size_t)B * H * 2, "tap h1")) != A8W8_OK) return st;

    // post-attention RMSNorm, Gate/Up + SwiGLU
    e = launch_rmsnorm_rows(hidden, B, H, reinterpret_cast<const bf16*>(w->post_norm_w), c.rms_eps,
                            xn, L);
    if (e != cudaSuccess) return cuda_fail(e, "post-attention RMSNorm");
    if ((st = tap(T.hn, xn, (size_t)B * H * 2, "tap hn")) != A8W8_OK) return st;
    g = Bf16GemvParams{};
    g.x = xn;
    g.ldx = H;
    g.W = reinterpret_cast<const bf16*>(w->w_gate_up);
    g.K = H;
    g.N = I;
    g.M = B;
    g.y = act;
    g.ldy = I;
    e = launch_bf16_gemv(g, true, L);
    if (e != cudaSuccess) return cuda_fail(e, "Gate/Up projection");
    if ((st = tap(T.act, act, (size_t)B * I * 2, "tap act")) != A8W8_OK) return st;

    // down projection + residual (in place)
    g = Bf16GemvParams{};
    g.x = act;
    g.ldx = I;
    g.W = reinterpret_cast<const bf16*>(w->w_down);
    g.K = I;
    g.N = H;
    g.M = B;
    g.residual = hidden;
    g.y = hidden;
    g.ldy = H;
    e = launch_bf16_gemv(g, false, L);
    if (e != cudaSuccess) return cuda_fail(e, "down projection");
    return A8W8_OK;
}

a8w8_status check_layer_common(const a8w8_config* cfg, int B, int max_blocks, int num_blocks,
                               const float* rope, int max_pos) {
    a8w8_status s = check_config(cfg);
    if (s != A8W8_OK) return s;
    if (B < 1 || B > 64) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "B=%d outside [1, 64]", B);
    if (max_blocks < 1 || num_blocks < 1)
        return fail(A8W8_ERR_INVALID_ARG, "max_blocks and num_blocks must be >= 1");
    if ((long long)max_blocks * cfg->page_size > (1 << 24))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "context longer than 2^24 tokens");
    if (!rope || max_pos < 1) return fail(A8W8_ERR_INVALID_ARG, "rope table missing");
    return A8W8_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================

extern "C" {

const char* a8w8_last_error(void) { return g_last_error.c_str(); }

int a8w8_version(void) { return 100; }

a8w8_status a8w8_read_device_errors(unsigned* bits, void* stream) {
    if (!bits) return fail(A8W8_ERR_INVALID_ARG, "bits is NULL");
    CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize");
    unsigned* w = device_error_word();
    if (!w) return fail(A8W8_ERR_CUDA, "device error word unavailable");
    unsigned h = 0;
    CUDA_TRY(cudaMemcpy(&h, w, sizeof h, cudaMemcpyDeviceToHost), "read device error word");
    CUDA_TRY(cudaMemset(w, 0, sizeof h), "clear device error word");
    *bits = h;
    return A8W8_OK;
}

a8w8_status a8w8_quant_rows(const a8w8_bf16* x, int rows, int cols, int ldx, int8_t* q,
                            float* row_scale, void* stream) {
    if (rows < 0 || cols < 0) return fail(A8W8_ERR_INVALID_ARG, "negative size");
    if (rows == 0) return A8W8_OK;
    if (cols == 0 || cols % 8 || ldx % 8 || ldx < cols)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "cols and ldx must be positive multiples of 8, ldx >= cols");
    a8w8_status s = check_ptrs({x, q, row_scale}, "a8w8_quant_rows");
    if (s != A8W8_OK) return s;
    cudaError_t e = launch_quant_rows(reinterpret_cast<const bf16*>(x), rows, cols, ldx, q, row_scale,
                                      make_launch(stream, false));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "a8w8_quant_rows");
}

static a8w8_status linear_common(const int8_t* xq, const float* x_scale, int M, int K,
                                 const int8_t* W, const float* w_scale, int N, int k_splits,
                                 const a8w8_bf16* residual, a8w8_bf16* y, int32_t* acc_out,
                                 bool swiglu, void* stream, const char* name) {
    if (M < 0 || K < 0 || N < 0) return fail(A8W8_ERR_INVALID_ARG, "%s: negative size", name);
    if (M == 0 || N == 0) return A8W8_OK;
    if (K == 0 || K % 16) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "%s: K must be a positive multiple of 16", name);
    if (k_splits != 1 && k_splits != 2) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "%s: k_splits must be 1 or 2", name);
    if ((K / k_splits) % 16 || K % k_splits)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "%s: K / k_splits must be a multiple of 16", name);
    a8w8_status s = check_ptrs({xq, x_scale, W, w_scale, y}, name);
    if (s != A8W8_OK) return s;
    if (residual && !aligned16(residual)) return fail(A8W8_ERR_INVALID_ARG, "%s: residual misaligned", name);
    Launch L = make_launch(stream, false);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "%s: no CUDA device", name);
    GemvParams g = {};
    g.W = W;
    g.w_scale = w_scale;
    g.K = K;
    g.N = N;
    g.xq = xq;
    g.x_scale = x_scale;
    g.residual = reinterpret_cast<const bf16*>(residual);
    g.y = reinterpret_cast<bf16*>(y);
    g.ldy = N;
    g.acc_out = acc_out;
    cudaError_t e = run_gemv(PRO_I8, swiglu ? EPI_SWIGLU : EPI_STORE, k_splits, g, M, L);
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, name);
}

a8w8_status a8w8_linear(const int8_t* xq, const float* x_scale, int M, int K, const int8_t* W,
                        const float* w_scale, int N, int k_splits, const a8w8_bf16* residual,
                        a8w8_bf16* y, int32_t* acc_out, void* stream) {
    return linear_common(xq, x_scale, M, K, W, w_scale, N, k_splits, residual, y, acc_out, false,
                         stream, "a8w8_linear");
}

a8w8_status a8w8_gate_up_swiglu(const int8_t* xq, const float* x_scale, int M, int K,
                                const int8_t* W_gu, const float* s_gu, int I, a8w8_bf16* act,
                                int32_t* acc_out, void* stream) {
    return linear_common(xq, x_scale, M, K, W_gu, s_gu, I, 1, nullptr, act, acc_out, true, stream,
                         "a8w8_gate_up_swiglu");
}

a8w8_status a8w8_matmul_i8(const int8_t* xq, int M, int K, const int8_t* W, int N, int k0, int k1,
                           int32_t* acc, void* scratch, void* stream) {
    const char* name = "a8w8_matmul_i8";
    if (M < 0 || N < 0 || K < 0) return fail(A8W8_ERR_INVALID_ARG, "%s: negative size", name);
    if (M == 0 || N == 0) return A8W8_OK;
    if (K == 0 || K % 64 || k0 < 0 || k1 > K || k0 % 64 || (k1 - k0) <= 0 || (k1 - k0) % 64)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE,
                    "%s: K, k0 and k1 - k0 must be positive multiples of 64 with k1 <= K", name);
    a8w8_status s = check_ptrs({xq, W, acc, scratch}, name);
    if (s != A8W8_OK) return s;
    Launch L = make_launch(stream, false);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "%s: no CUDA device", name);
    uint16_t* x16 = static_cast<uint16_t*>(scratch);
    cudaError_t e = launch_i8_to_f16(xq, (size_t)M * K, x16, L);
    if (e == cudaSuccess) e = launch_gemm_tc(x16, M, W, N, K, k0, k1, acc, N, device_error_word(), L);
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, name);
}

a8w8_status a8w8_rmsnorm_gate_up_swiglu(const a8w8_bf16* x, int M, int K,
                                        const a8w8_bf16* norm_w, float eps, const int8_t* W_gu,
                                        const float* s_gu, int I, a8w8_bf16* act, void* stream) {
    const char* name = "a8w8_rmsnorm_gate_up_swiglu";
    if (M < 0 || K < 0 || I < 0) return fail(A8W8_ERR_INVALID_ARG, "%s: negative size", name);
    if (M == 0 || I == 0) return A8W8_OK;
    if (K == 0 || K % 16 || K > 65536)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "%s: K must be a positive multiple of 16, at most 65536", name);
    if (!(eps >= 0.0f)) return fail(A8W8_ERR_INVALID_ARG, "%s: eps must be >= 0", name);
    a8w8_status s = check_ptrs({x, norm_w, W_gu, s_gu, act}, name);
    if (s != A8W8_OK) return s;
    Launch L = make_launch(stream, false);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "%s: no CUDA device", name);
    GemvParams g = {};
    g.W = W_gu;
    g.w_scale = s_gu;
    g.K = K;
    g.N = I;
    g.x = reinterpret_cast<const bf16*>(x);
    g.ldx = K;
    g.norm_w = reinterpret_cast<const bf16*>(norm_w);
    g.eps = eps;
    g.y = reinterpret_cast<bf16*>(act);
    g.ldy = I;
    // no code buffers: every batch tile runs the streaming kernel with the
    // normalisation and quantisation in its prologue, as the decode layer
    // does for one or two rows
    cudaError_t e = run_gemv(PRO_NORM_QUANT, EPI_SWIGLU, 1, g, M, L);
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, name);
}

a8w8_status paged_kv_write(const a8w8_bf16* k, const a8w8_bf16* v, int T, int Hkv, int D,
                           const int32_t* slot_mapping, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                           int num_blocks, int page_size, void* stream) {
    if (T < 0 || Hkv <= 0 || D <= 0 || num_blocks < 0 || page_size <= 0)
        return fail(A8W8_ERR_INVALID_ARG, "paged_kv_write: bad size");
    if (T == 0) return A8W8_OK;
    if ((Hkv * D) % 8) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "paged_kv_write: Hkv*D must be a multiple of 8");
    a8w8_status s = check_ptrs({k, v, slot_mapping, k_cache, v_cache}, "paged_kv_write");
    if (s != A8W8_OK) return s;
    cudaError_t e = launch_kv_write(reinterpret_cast<const bf16*>(k), reinterpret_cast<const bf16*>(v), T,
                                    Hkv, D, slot_mapping, reinterpret_cast<bf16*>(k_cache),
                                    reinterpret_cast<bf16*>(v_cache), (long)num_blocks * page_size,
                                    device_error_word(), make_launch(stream, false));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "paged_kv_write");
}

size_t a8w8_attention_workspace_bytes(int B, int Hq, int D, int max_ctx) {
    if (B <= 0 || Hq <= 0 || D <= 0 || max_ctx <= 0) return 0;
    return attn_part_bytes(B, Hq, D, max_ctx, false);
}

a8w8_status paged_decode_attention_bf16(const a8w8_bf16* q, const a8w8_bf16* k_cache,
                                        const a8w8_bf16* v_cache, const int32_t* block_table,
                                        const int32_t* ctx_lens, int B, int Hq, int Hkv, int D,
                                        int page_size, int max_blocks, int num_blocks,
                                        float softmax_scale, a8w8_bf16* out, void* ws,
                                        size_t ws_bytes, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || page_size <= 0 || max_blocks <= 0 || num_blocks <= 0)
        return fail(A8W8_ERR_INVALID_ARG, "paged_decode_attention_bf16: bad size");
    if (B == 0) return A8W8_OK;
    if (D != 64 && D != 128) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "head_dim %d not supported", D);
    if (Hq % Hkv || Hq / Hkv > 8) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "Hq/Hkv must be an integer <= 8");
    if ((long long)max_blocks * page_size > (1 << 24))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "context longer than 2^24 tokens");
    a8w8_status s = check_ptrs({q, k_cache, v_cache, block_table, ctx_lens, out}, "paged_decode_attention_bf16");
    if (s != A8W8_OK) return s;
    const size_t need = attn_part_bytes(B, Hq, D, max_blocks * page_size, false);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
        return fail(A8W8_ERR_WORKSPACE, "attention workspace needs %zu bytes", need);
    AttnParams a = {};
    a.q = reinterpret_cast<const bf16*>(q);
    a.q_stride = Hq * D;
    a.fused = false;
    a.k_cache = const_cast<bf16*>(reinterpret_cast<const bf16*>(k_cache));
    a.v_cache = const_cast<bf16*>(reinterpret_cast<const bf16*>(v_cache));
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = page_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.scale = softmax_scale;
    a.out = reinterpret_cast<bf16*>(out);
    a.part = static_cast<float*>(ws);
    a.err = device_error_word();
    cudaError_t e = launch_attention(a, make_launch(stream, false));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "paged_decode_attention_bf16");
}

a8w8_status paged_kv_write_i8(const a8w8_bf16* k, const a8w8_bf16* v, int T, int Hkv, int D,
                              const int32_t* slot_mapping, int8_t* k_codes, int8_t* v_codes,
                              float* k_scale, float* v_scale, int num_blocks, int page_size,
                              void* stream) {
    if (T < 0 || Hkv <= 0 || num_blocks < 0 || page_size <= 0)
        return fail(A8W8_ERR_INVALID_ARG, "paged_kv_write_i8: bad size");
    if (T == 0) return A8W8_OK;
    if (D != 64 && D != 128) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "paged_kv_write_i8: head_dim %d not supported", D);
    a8w8_status s = check_ptrs({k, v, slot_mapping, k_codes, v_codes, k_scale, v_scale}, "paged_kv_write_i8");
    if (s != A8W8_OK) return s;
    cudaError_t e = launch_kv_write_i8(reinterpret_cast<const bf16*>(k), reinterpret_cast<const bf16*>(v),
                                       T, Hkv, D, slot_mapping, k_codes, v_codes, k_scale, v_scale,
                                       (long)num_blocks * page_size, device_error_word(),
                                       make_launch(stream, false));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "paged_kv_write_i8");
}

a8w8_status paged_decode_attention_i8kv(const a8w8_bf16* q, const int8_t* k_codes,
                                        const int8_t* v_codes, const float* k_scale,
                                        const float* v_scale, const int32_t* block_table,
                                        const int32_t* ctx_lens, int B, int Hq, int Hkv, int D,
                                        int page_size, int max_blocks, int num_blocks,
                                        float softmax_scale, a8w8_bf16* out, void* ws,
                                        size_t ws_bytes, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || page_size <= 0 || max_blocks <= 0 || num_blocks <= 0)
        return fail(A8W8_ERR_INVALID_ARG, "paged_decode_attention_i8kv: bad size");
    if (B == 0) return A8W8_OK;
    if (D != 64 && D != 128) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "head_dim %d not supported", D);
    if (Hq % Hkv || Hq / Hkv > 8) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "Hq/Hkv must be an integer <= 8");
    if ((long long)max_blocks * page_size > (1 << 24))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "context longer than 2^24 tokens");
    a8w8_status s = check_ptrs({q, k_codes, v_codes, k_scale, v_scale, block_table, ctx_lens, out},
                               "paged_decode_attention_i8kv");
    if (s != A8W8_OK) return s;
    const size_t need = attn_part_bytes(B, Hq, D, max_blocks * page_size, false);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
        return fail(A8W8_ERR_WORKSPACE, "attention workspace needs %zu bytes", need);
    AttnI8Params ai = {};
    AttnParams& a = ai.a;
    a.q = reinterpret_cast<const bf16*>(q);
    a.q_stride = Hq * D;
    a.fused = false;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = page_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.scale = softmax_scale;
    a.out = reinterpret_cast<bf16*>(out);
    a.part = static_cast<float*>(ws);
    a.err = device_error_word();
    ai.k_codes = const_cast<int8_t*>(k_codes);
    ai.v_codes = const_cast<int8_t*>(v_codes);
    ai.k_scale = const_cast<float*>(k_scale);
    ai.v_scale = const_cast<float*>(v_scale);
    cudaError_t e = launch_attention_i8(ai, make_launch(stream, false));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "paged_decode_attention_i8kv");
}

}  // extern "C"

// Scratch of paged_decode_attention_bf16_noalloc: a fixed device array owned by
// the library, so that callers with no way to allocate device memory can run
// split-KV attention. Host code must not pass the array's name to a kernel (on
// the host it is only a stand-in); the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float g_noalloc_attn_scratch[A8W8_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

// Device address of the scratch array in the current context (looked up on
// the first use in each context, under the library's lock), or nullptr with
// the error message set.
float* noalloc_scratch_address() {
    void* p = symbol_address(g_noalloc_attn_scratch);
    if (!p) {
        fail(A8W8_ERR_CUDA, "paged_decode_attention_bf16_noalloc: scratch address lookup failed");
        return nullptr;
    }
    return static_cast<float*>(p);
}

}  // namespace

extern "C" {

a8w8_status paged_decode_attention_bf16_noalloc(const a8w8_bf16* q, const a8w8_bf16* k_cache,
                                                const a8w8_bf16* v_cache,
                                                const int32_t* block_table,
                                                const int32_t* ctx_lens, int B, int Hq, int Hkv,
                                                int D, int page_size, int max_blocks,
                                                int num_blocks, float softmax_scale,
                                                a8w8_bf16* out, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || page_size <= 0 || max_blocks <= 0 || num_blocks <= 0)
        return fail(A8W8_ERR_INVALID_ARG, "paged_decode_attention_bf16_noalloc: bad size");
    if (B == 0) return A8W8_OK;
    if (D != 64 && D != 128) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "head_dim %d not supported", D);
    if (Hq % Hkv || Hq / Hkv > 8) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "Hq/Hkv must be an integer <= 8");
    if ((long long)max_blocks * page_size > (1 << 24))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "context longer than 2^24 tokens");
    a8w8_status s = check_ptrs({q, k_cache, v_cache, block_table, ctx_lens, out},
                               "paged_decode_attention_bf16_noalloc");
    if (s != A8W8_OK) return s;
    const size_t need = attn_part_bytes(B, Hq, D, max_blocks * page_size, false);
    if (need > A8W8_NOALLOC_SCRATCH_BYTES)
        return fail(A8W8_ERR_WORKSPACE,
                    "paged_decode_attention_bf16_noalloc: split-KV partials need %zu bytes, more than "
                    "the %zu-byte built-in scratch; use paged_decode_attention_bf16 with a workspace",
                    need, (size_t)A8W8_NOALLOC_SCRATCH_BYTES);
    float* scratch = nullptr;
    if (need > 0) {
        scratch = noalloc_scratch_address();
        if (!scratch) return A8W8_ERR_CUDA;
    }
    AttnParams a = {};
    a.q = reinterpret_cast<const bf16*>(q);
    a.q_stride = Hq * D;
    a.fused = false;
    a.k_cache = const_cast<bf16*>(reinterpret_cast<const bf16*>(k_cache));
    a.v_cache = const_cast<bf16*>(reinterpret_cast<const bf16*>(v_cache));
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.page = page_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.scale = softmax_scale;
    a.out = reinterpret_cast<bf16*>(out);
    a.part = scratch;
    a.err = device_error_word();
    cudaError_t e = launch_attention(a, make_launch(stream, false));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "paged_decode_attention_bf16_noalloc");
}

a8w8_status a8w8_rope_table(float* rope, int max_pos, int D, double theta, void* stream) {
    if (max_pos < 0 || D <= 0 || D % 2 || D > 2048 || !(theta > 0.0))
        return fail(A8W8_ERR_INVALID_ARG, "a8w8_rope_table: bad arguments");
    if (max_pos == 0) return A8W8_OK;
    a8w8_status s = check_ptrs({rope}, "a8w8_rope_table");
    if (s != A8W8_OK) return s;
    cudaError_t e = launch_rope_table(rope, max_pos, D, theta, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "a8w8_rope_table");
}

size_t a8w8_sample_workspace_bytes(int B, int V) {
    if (B <= 0 || V <= 0) return 0;
    return sample_workspace_bytes(B, V);
}

a8w8_status a8w8_sample(const float* logits, int B, int V, int ld, float temperature, float top_p,
                        uint64_t seed, uint64_t step, int32_t* next_tokens, void* ws,
                        size_t ws_bytes, void* stream) {
    if (B < 0 || V < 1 || ld < V) return fail(A8W8_ERR_INVALID_ARG, "sample: need B >= 0, V >= 1, ld >= V");
    if (!(top_p > 0.0f && top_p <= 1.0f)) return fail(A8W8_ERR_INVALID_ARG, "sample: top_p must be in (0, 1]");
    if (temperature != temperature || temperature > 3.0e38f)
        return fail(A8W8_ERR_INVALID_ARG, "sample: temperature must be finite");
    if (B == 0) return A8W8_OK;
    if (!logits || !next_tokens) return fail(A8W8_ERR_INVALID_ARG, "sample: NULL pointer");
    if (!ws || ws_bytes < sample_workspace_bytes(B, V) || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "sample: needs %zu bytes of workspace",
                    sample_workspace_bytes(B, V));
    Launch L = make_launch(stream, true);
    CUDA_TRY(launch_sample(logits, B, V, ld, temperature, top_p, seed, step,
                           static_cast<float*>(ws), next_tokens, L),
             "sample");
    return A8W8_OK;
}

size_t a8w8_workspace_bytes(const a8w8_config* cfg, int max_B, int max_blocks) {
    if (!cfg || max_B <= 0 || max_blocks <= 0) return 0;
    return ws_layout(*cfg, max_B, max_blocks).total;
}

a8w8_status a8w8_decode_layer(const a8w8_layer_weights* w, const a8w8_config* cfg, int B,
                              a8w8_bf16* hidden, const int32_t* slot_mapping,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* ctx_lens, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                              const float* rope, int max_pos, void* ws, size_t ws_bytes,
                              const a8w8_layer_taps* taps, void* stream) {
    a8w8_status s = check_layer_common(cfg, B, max_blocks, num_blocks, rope, max_pos);
    if (s != A8W8_OK) return s;
    if ((s = check_layer_weights(w)) != A8W8_OK) return s;
    if ((s = check_ptrs({hidden, slot_mapping, block_table, ctx_lens, k_cache, v_cache, rope},
                        "a8w8_decode_layer")) != A8W8_OK)
        return s;
    const WsLayout lay = ws_layout(*cfg, B, max_blocks);
    if (!ws || ws_bytes < lay.total || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "decode layer workspace needs %zu bytes", lay.total);
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    return enqueue_layer(w, *cfg, B, reinterpret_cast<bf16*>(hidden), slot_mapping, block_table,
                         max_blocks, num_blocks, ctx_lens, reinterpret_cast<bf16*>(k_cache),
                         reinterpret_cast<bf16*>(v_cache), rope, max_pos,
                         static_cast<unsigned char*>(ws), lay, taps, L);
}

a8w8_status a8w8_decode_layer_i8kv(const a8w8_layer_weights* w, const a8w8_config* cfg, int B,
                                   a8w8_bf16* hidden, const int32_t* slot_mapping,
                                   const int32_t* block_table, int max_blocks, int num_blocks,
                                   const int32_t* ctx_lens, int8_t* k_codes, int8_t* v_codes,
                                   float* k_scale, float* v_scale, const float* rope, int max_pos,
                                   void* ws, size_t ws_bytes, const a8w8_layer_taps* taps,
                                   void* stream) {
    a8w8_status s = check_layer_common(cfg, B, max_blocks, num_blocks, rope, max_pos);
    if (s != A8W8_OK) return s;
    if ((s = check_layer_weights(w)) != A8W8_OK) return s;
    if ((s = check_ptrs({hidden, slot_mapping, block_table, ctx_lens, k_codes, v_codes, k_scale,
                         v_scale, rope},
                        "a8w8_decode_layer_i8kv")) != A8W8_OK)
        return s;
    const WsLayout lay = ws_layout(*cfg, B, max_blocks);
    if (!ws || ws_bytes < lay.total || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "decode layer workspace needs %zu bytes", lay.total);
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    const KvI8 kv8 = {k_codes, v_codes, k_scale, v_scale};
    return enqueue_layer(w, *cfg, B, reinterpret_cast<bf16*>(hidden), slot_mapping, block_table,
                         max_blocks, num_blocks, ctx_lens, nullptr, nullptr, rope, max_pos,
                         static_cast<unsigned char*>(ws), lay, taps, L, false, &kv8);
}

a8w8_status bf16_linear(const a8w8_bf16* x, int M, int K, const a8w8_bf16* W, int N,
                        const a8w8_bf16* residual, a8w8_bf16* y, void* stream) {
    if (M < 0 || K < 0 || N < 0) return fail(A8W8_ERR_INVALID_ARG, "bf16_linear: negative size");
    if (M == 0 || N == 0) return A8W8_OK;
    if (K == 0 || K % 8 || bf16_gemv_batch_tile(K) == 0)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "bf16_linear: K must be a positive multiple of 8, at most 49152");
    a8w8_status s = check_ptrs({x, W, y}, "bf16_linear");
    if (s != A8W8_OK) return s;
    if (residual && !aligned16(residual)) return fail(A8W8_ERR_INVALID_ARG, "bf16_linear: residual misaligned");
    Launch L = make_launch(stream, false);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "bf16_linear: no CUDA device");
    Bf16GemvParams g = {};
    g.x = reinterpret_cast<const bf16*>(x);
    g.ldx = K;
    g.W = reinterpret_cast<const bf16*>(W);
    g.K = K;
    g.N = N;
    g.M = M;
    g.residual = reinterpret_cast<const bf16*>(residual);
    g.y = reinterpret_cast<bf16*>(y);
    g.ldy = N;
    cudaError_t e = launch_bf16_gemv(g, false, L);
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "bf16_linear");
}

a8w8_status bf16_gate_up_swiglu(const a8w8_bf16* x, int M, int K, const a8w8_bf16* W_gu, int I,
                                a8w8_bf16* act, void* stream) {
    if (M < 0 || K < 0 || I < 0) return fail(A8W8_ERR_INVALID_ARG, "bf16_gate_up_swiglu: negative size");
    if (M == 0 || I == 0) return A8W8_OK;
    if (K == 0 || K % 8 || bf16_gemv_batch_tile(K) == 0)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "bf16_gate_up_swiglu: K must be a positive multiple of 8, at most 49152");
    a8w8_status s = check_ptrs({x, W_gu, act}, "bf16_gate_up_swiglu");
    if (s != A8W8_OK) return s;
    Launch L = make_launch(stream, false);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "bf16_gate_up_swiglu: no CUDA device");
    Bf16GemvParams g = {};
    g.x = reinterpret_cast<const bf16*>(x);
    g.ldx = K;
    g.W = reinterpret_cast<const bf16*>(W_gu);
    g.K = K;
    g.N = I;
    g.M = M;
    g.y = reinterpret_cast<bf16*>(act);
    g.ldy = I;
    cudaError_t e = launch_bf16_gemv(g, true, L);
    return e == cudaSuccess ? A8W8_OK : cuda_fail(e, "bf16_gate_up_swiglu");
}

a8w8_status bf16_decode_layer(const a8w8_bf16_layer_weights* w, const a8w8_config* cfg, int B,
                              a8w8_bf16* hidden, const int32_t* slot_mapping,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* ctx_lens, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                              const float* rope, int max_pos, void* ws, size_t ws_bytes,
                              const a8w8_layer_taps* taps, void* stream) {
    a8w8_status s = check_layer_common(cfg, B, max_blocks, num_blocks, rope, max_pos);
    if (s != A8W8_OK) return s;
    if (!w) return fail(A8W8_ERR_INVALID_ARG, "layer weights are NULL");
    if ((s = check_ptrs({w->input_norm_w, w->w_qkv, w->q_norm_w, w->k_norm_w, w->w_o,
                         w->post_norm_w, w->w_gate_up, w->w_down},
                        "BF16 layer weights")) != A8W8_OK)
        return s;
    const int D = cfg->head_dim;
    const int kmax = std::max({cfg->hidden, cfg->num_q_heads * D, cfg->intermediate});
    if (bf16_gemv_batch_tile(kmax) == 0)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "bf16_decode_layer: projection K above 49152");
    if ((s = check_ptrs({hidden, slot_mapping, block_table, ctx_lens, k_cache, v_cache, rope},
                        "bf16_decode_layer")) != A8W8_OK)
        return s;
    const WsLayout lay = ws_layout(*cfg, B, max_blocks);
    if (!ws || ws_bytes < lay.total || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "decode layer workspace needs %zu bytes", lay.total);
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    return enqueue_bf16_layer(w, *cfg, B, reinterpret_cast<bf16*>(hidden), slot_mapping,
                              block_table, max_blocks, num_blocks, ctx_lens,
                              reinterpret_cast<bf16*>(k_cache), reinterpret_cast<bf16*>(v_cache),
                              rope, max_pos, static_cast<unsigned char*>(ws), lay, taps, L);
}

a8w8_status a8w8_prefill_layer(const a8w8_layer_weights* w, const a8w8_config* cfg, int M,
                               a8w8_bf16* hidden, const int32_t* slot_mapping,
                               const int32_t* block_table, int max_blocks, int num_blocks,
                               const int32_t* ctx_lens, a8w8_bf16* k_cache, a8w8_bf16* v_cache,
                               const float* rope, int max_pos, void* ws, size_t ws_bytes,
                               const a8w8_layer_taps* taps, void* stream) {
    if (M < 1 || M > 16384) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "M=%d outside [1, 16384]", M);
    a8w8_status s = check_layer_common(cfg, 1, max_blocks, num_blocks, rope, max_pos);
    if (s != A8W8_OK) return s;
    if ((s = check_layer_weights(w)) != A8W8_OK) return s;
    if ((s = check_ptrs({hidden, slot_mapping, block_table, ctx_lens, k_cache, v_cache, rope},
                        "a8w8_prefill_layer")) != A8W8_OK)
        return s;
    if (!attn_group_shape_ok(cfg->num_q_heads, cfg->num_kv_heads, cfg->head_dim,
                             max_blocks * cfg->page_size))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE,
                    "prefill attention needs Hq/Hkv <= 7 and at most 64 chunks of 128 tokens");
    const WsLayout lay = ws_layout(*cfg, M, max_blocks);
    if (!ws || ws_bytes < lay.total || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "prefill layer workspace needs %zu bytes", lay.total);
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    return enqueue_layer(w, *cfg, M, reinterpret_cast<bf16*>(hidden), slot_mapping, block_table,
                         max_blocks, num_blocks, ctx_lens, reinterpret_cast<bf16*>(k_cache),
                         reinterpret_cast<bf16*>(v_cache), rope, max_pos,
                         static_cast<unsigned char*>(ws), lay, taps, L, true);
}

a8w8_status a8w8_prefill_layer_i8kv(const a8w8_layer_weights* w, const a8w8_config* cfg, int M,
                                    a8w8_bf16* hidden, const int32_t* slot_mapping,
                                    const int32_t* block_table, int max_blocks, int num_blocks,
                                    const int32_t* ctx_lens, int8_t* k_codes, int8_t* v_codes,
                                    float* k_scale, float* v_scale, const float* rope,
                                    int max_pos, void* ws, size_t ws_bytes,
                                    const a8w8_layer_taps* taps, void* stream) {
    if (M < 1 || M > 16384) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "M=%d outside [1, 16384]", M);
    a8w8_status s = check_layer_common(cfg, 1, max_blocks, num_blocks, rope, max_pos);
    if (s != A8W8_OK) return s;
    if ((s = check_layer_weights(w)) != A8W8_OK) return s;
    if ((s = check_ptrs({hidden, slot_mapping, block_table, ctx_lens, k_codes, v_codes, k_scale,
                         v_scale, rope},
                        "a8w8_prefill_layer_i8kv")) != A8W8_OK)
        return s;
    if (!attn_group_shape_ok(cfg->num_q_heads, cfg->num_kv_heads, cfg->head_dim,
                             max_blocks * cfg->page_size))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE,
                    "prefill attention needs Hq/Hkv <= 7 and at most 64 chunks of 128 tokens");
    const WsLayout lay = ws_layout(*cfg, M, max_blocks);
    if (!ws || ws_bytes < lay.total || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "prefill layer workspace needs %zu bytes", lay.total);
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    const KvI8 kv8 = {k_codes, v_codes, k_scale, v_scale};
    return enqueue_layer(w, *cfg, M, reinterpret_cast<bf16*>(hidden), slot_mapping, block_table,
                         max_blocks, num_blocks, ctx_lens, nullptr, nullptr, rope, max_pos,
                         static_cast<unsigned char*>(ws), lay, taps, L, true, &kv8);
}

static a8w8_status check_step(const a8w8_model* m, const a8w8_config* cfg, int B, int max_blocks,
                              int num_blocks, a8w8_bf16* const* k_caches,
                              a8w8_bf16* const* v_caches, const float* rope, int max_pos,
                              size_t ws_bytes, const void* ws) {
    a8w8_status s = check_layer_common(cfg, B, max_blocks, num_blocks, rope, max_pos);
    if (s != A8W8_OK) return s;
    if (!m) return fail(A8W8_ERR_INVALID_ARG, "model is NULL");
    if (cfg->vocab <= 0 || cfg->num_layers < 1) return fail(A8W8_ERR_INVALID_ARG, "vocab and num_layers must be >= 1");
    if ((s = check_ptrs({m->embed, m->final_norm_w, m->lm_head}, "model")) != A8W8_OK) return s;
    if (!m->layers || !k_caches || !v_caches) return fail(A8W8_ERR_INVALID_ARG, "layer arrays are NULL");
    for (int l = 0; l < cfg->num_layers; ++l) {
        if ((s = check_layer_weights(&m->layers[l])) != A8W8_OK) return s;
        if ((s = check_ptrs({k_caches[l], v_caches[l]}, "KV caches")) != A8W8_OK) return s;
    }
    const WsLayout lay = ws_layout(*cfg, B, max_blocks);
    if (!ws || ws_bytes < lay.total || !aligned16(ws))
        return fail(A8W8_ERR_WORKSPACE, "decode step workspace needs %zu bytes", lay.total);
    return A8W8_OK;
}

// Sampling inside a captured step: the sampler runs on the step's logits and
// overwrites the argmax, reading its Philox step from `step` (advanced by one
// per step on the device).
struct StepSampling {
    float T, top_p;
    uint64_t seed;
    uint64_t* step;
    float* ws;
};

static a8w8_status enqueue_step(const a8w8_model* m, const a8w8_config& c, int B,
                                const int32_t* token_ids, const int32_t* slot_mapping,
                                const int32_t* block_table, int max_blocks, int num_blocks,
                                const int32_t* ctx_lens, a8w8_bf16* const* k_caches,
                                a8w8_bf16* const* v_caches, const float* rope, int max_pos,
                                int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                                unsigned char* ws, const Launch& L, bool device_loop,
                                const KvI8* kv8 = nullptr, const StepSampling* smp = nullptr) {
    // kv8: the layers' INT8 caches (num_layers entries) instead of k_caches /
    // v_caches; the per-operation kernels only
    const WsLayout lay = ws_layout(c, B, max_blocks);
    bf16* hidden = reinterpret_cast<bf16*>(ws + lay.hid);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(ws + lay.keys);
    unsigned* ticket = reinterpret_cast<unsigned*>(ws + lay.ticket);
    if (!kv8 && !smp && (c.flags & A8W8_FLAG_PERSISTENT_STEP) &&
        step_supported(B, c.head_dim, c.num_layers, c.hidden, c.intermediate, c.num_q_heads,
                       c.num_kv_heads, max_blocks * c.page_size, L.num_sms) &&
        c.down_k_splits == 2) {
        StepParams P;
        std::memset(&P, 0, sizeof P);
        P.B = B;
        P.H = c.hidden;
        P.Hq = c.num_q_heads;
        P.Hkv = c.num_kv_heads;
        P.D = c.head_dim;
        P.I = c.intermediate;
        P.vocab = c.vocab;
        P.page = c.page_size;
        P.max_blocks = max_blocks;
        P.num_blocks = num_blocks;
        P.max_pos = max_pos;
        P.L = c.num_layers;
        P.down_splits = c.down_k_splits;
        P.device_loop = device_loop ? 1 : 0;
        P.eps = c.rms_eps;
        {
            const double sd = 1.0 / std::sqrt((double)c.head_dim);
            P.attn_scale = (float)sd;
            P.attn_scale_lo = (float)(sd - (double)P.attn_scale);
        }
        P.embed = reinterpret_cast<const bf16*>(m->embed);
        P.final_norm_w = reinterpret_cast<const bf16*>(m->final_norm_w);
        P.lm_head = reinterpret_cast<const bf16*>(m->lm_head);
        P.rope = rope;
        P.token_ids = const_cast<int32_t*>(token_ids);
        P.slot_mapping = const_cast<int32_t*>(slot_mapping);
        P.block_table = const_cast<int32_t*>(block_table);
        P.ctx_lens = const_cast<int32_t*>(ctx_lens);
        P.next_tokens = next_tokens;
        P.logits = logits;
        P.final_hidden = reinterpret_cast<bf16*>(final_hidden);
        P.hidden = hidden;
        P.qkv = reinterpret_cast<bf16*>(ws + lay.qkv);
        P.attn = reinterpret_cast<bf16*>(ws + lay.attn);
        P.act = reinterpret_cast<bf16*>(ws + lay.act);
        P.part = reinterpret_cast<float*>(ws + lay.part);
        P.keys = keys;
        P.ticket = ticket;
        P.bar = reinterpret_cast<unsigned*>(ws + lay.bar);
        P.err = device_error_word();
        for (int l = 0; l < c.num_layers; ++l) {
            const a8w8_layer_weights& w = m->layers[l];
            StepLayer& d = P.layers[l];
            d.input_norm_w = reinterpret_cast<const bf16*>(w.input_norm_w);
            d.w_qkv = w.w_qkv;
            d.s_qkv = w.s_qkv;
            d.q_norm_w = reinterpret_cast<const bf16*>(w.q_norm_w);
            d.k_norm_w = reinterpret_cast<const bf16*>(w.k_norm_w);
            d.w_o = w.w_o;
            d.s_o = w.s_o;
            d.post_norm_w = reinterpret_cast<const bf16*>(w.post_norm_w);
            d.w_gate_up = w.w_gate_up;
            d.s_gate_up = w.s_gate_up;
            d.w_down = w.w_down;
            d.s_down = w.s_down;
            P.k_cache[l] = reinterpret_cast<bf16*>(k_caches[l]);
            P.v_cache[l] = reinterpret_cast<bf16*>(v_caches[l]);
        }
        cudaError_t e = cudaMemsetAsync(P.bar, 0, 16, L.stream);
        if (e != cudaSuccess) return cuda_fail(e, "step barrier reset");
        e = launch_step(P, L);
        if (e != cudaSuccess) return cuda_fail(e, "persistent decode step");
        return A8W8_OK;
    }
    cudaError_t e = launch_embed(reinterpret_cast<const bf16*>(m->embed), c.vocab, c.hidden,
                                 token_ids, B, hidden, keys, ticket, device_error_word(), L);
    if (e != cudaSuccess) return cuda_fail(e, "embedding");
    for (int l = 0; l < c.num_layers; ++l) {
        a8w8_status s = kv8
            ? enqueue_layer(&m->layers[l], c, B, hidden, slot_mapping, block_table, max_blocks,
                            num_blocks, ctx_lens, nullptr, nullptr, rope, max_pos, ws, lay, nullptr, L,
                            false, &kv8[l])
            : enqueue_layer(&m->layers[l], c, B, hidden, slot_mapping, block_table, max_blocks,
                            num_blocks, ctx_lens, reinterpret_cast<bf16*>(k_caches[l]),
                            reinterpret_cast<bf16*>(v_caches[l]), rope, max_pos, ws, lay,
                            nullptr, L);
        if (s != A8W8_OK) return s;
    }
    const int tile = lmhead_max_batch_tile();
    for (int b0 = 0; b0 < B; b0 += tile) {
        LmHeadParams p = {};
        p.hidden = hidden + (size_t)b0 * c.hidden;
        p.norm_w = reinterpret_cast<const bf16*>(m->final_norm_w);
        p.eps = c.rms_eps;
        p.W = reinterpret_cast<const bf16*>(m->lm_head);
        p.H = c.hidden;
        p.V = c.vocab;
        p.M = B - b0 < tile ? B - b0 : tile;
        p.logits = logits ? logits + (size_t)b0 * c.vocab : nullptr;
        p.final_hidden = final_hidden ? reinterpret_cast<bf16*>(final_hidden) + (size_t)b0 * c.hidden : nullptr;
        p.keys = keys + b0;
        p.ticket = ticket;
        p.next_tokens = next_tokens + b0;
        e = launch_lmhead_argmax(p, L);
        if (e != cudaSuccess) return cuda_fail(e, "LM head");
    }
    if (smp) {
        e = launch_sample(logits, B, c.vocab, c.vocab, smp->T, smp->top_p, smp->seed, 0, smp->ws,
                          next_tokens, L, smp->step);
        if (e != cudaSuccess) return cuda_fail(e, "sampling");
    }
    if (device_loop) {
        e = launch_advance(const_cast<int32_t*>(token_ids), const_cast<int32_t*>(slot_mapping),
                           block_table, const_cast<int32_t*>(ctx_lens), next_tokens, B, max_blocks,
                           c.page_size, L);
        if (e != cudaSuccess) return cuda_fail(e, "advance kernel");
    }
    return A8W8_OK;
}

a8w8_status a8w8_prefill_step(const a8w8_model* m, const a8w8_config* cfg, int M,
                              const int32_t* token_ids, const int32_t* slot_mapping,
                              const int32_t* block_table, int max_blocks, int num_blocks,
                              const int32_t* ctx_lens, a8w8_bf16* const* k_caches,
                              a8w8_bf16* const* v_caches, const float* rope, int max_pos, int S,
                              const int32_t* last_rows, int32_t* next_tokens, float* logits,
                              void* ws, size_t ws_bytes, void* stream) {
    if (M < 1 || M > 16384) return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "M=%d outside [1, 16384]", M);
    if (S < 1 || S > M) return fail(A8W8_ERR_INVALID_ARG, "S=%d outside [1, M]", S);
    // the model and caches as for a decode step of one row; the workspace for M rows
    a8w8_status s = check_step(m, cfg, 1, max_blocks, num_blocks, k_caches, v_caches, rope,
                               max_pos, ~(size_t)0, ws);
    if (s != A8W8_OK) return s;
    const int H = cfg->hidden, NQKV = (cfg->num_q_heads + 2 * cfg->num_kv_heads) * cfg->head_dim;
    if (!attn_group_shape_ok(cfg->num_q_heads, cfg->num_kv_heads, cfg->head_dim,
                             max_blocks * cfg->page_size))
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE,
                    "prefill attention needs Hq/Hkv <= 7 and at most 64 chunks of 128 tokens");
    if (cfg->intermediate < H && NQKV < H)
        return fail(A8W8_ERR_UNSUPPORTED_SHAPE, "prefill step needs intermediate or QKV width >= hidden");
    if ((s = check_ptrs({token_ids, slot_mapping, block_table, ctx_lens, last_rows, next_tokens},
                        "a8w8_prefill_step")) != A8W8_OK)
        return s;
    if (logits && !aligned16(logits)) return fail(A8W8_ERR_INVALID_ARG, "logits misaligned");
    const WsLayout lay = ws_layout(*cfg, M, max_blocks);
    if (ws_bytes < lay.total) return fail(A8W8_ERR_WORKSPACE, "prefill step workspace needs %zu bytes", lay.total);
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    const a8w8_config& c = *cfg;
    unsigned char* w = static_cast<unsigned char*>(ws);
    bf16* hidden = reinterpret_cast<bf16*>(w + lay.hid);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(w + lay.keys);
    unsigned* ticket = reinterpret_cast<unsigned*>(w + lay.ticket);
    cudaError_t e = launch_embed(reinterpret_cast<const bf16*>(m->embed), c.vocab, H, token_ids, M,
                                 hidden, keys, ticket, device_error_word(), L);
    if (e != cudaSuccess) return cuda_fail(e, "embedding");
    for (int l = 0; l < c.num_layers; ++l) {
        s = enqueue_layer(&m->layers[l], c, M, hidden, slot_mapping, block_table, max_blocks,
                          num_blocks, ctx_lens, reinterpret_cast<bf16*>(k_caches[l]),
                          reinterpret_cast<bf16*>(v_caches[l]), rope, max_pos, w, lay, nullptr, L,
                          true);
        if (s != A8W8_OK) return s;
    }
    // the last rows into a dense block (the SwiGLU or QKV buffer, free by now)
    bf16* last = reinterpret_cast<bf16*>(w + (c.intermediate >= H ? lay.act : lay.qkv));
    e = launch_gather_rows(hidden, H, last_rows, S, M, last, device_error_word(), L);
    if (e != cudaSuccess) return cuda_fail(e, "gather last rows");
    const int tile = lmhead_max_batch_tile();
    for (int b0 = 0; b0 < S; b0 += tile) {
        LmHeadParams p = {};
        p.hidden = last + (size_t)b0 * H;
        p.norm_w = reinterpret_cast<const bf16*>(m->final_norm_w);
        p.eps = c.rms_eps;
        p.W = reinterpret_cast<const bf16*>(m->lm_head);
        p.H = H;
        p.V = c.vocab;
        p.M = S - b0 < tile ? S - b0 : tile;
        p.logits = logits ? logits + (size_t)b0 * c.vocab : nullptr;
        p.final_hidden = nullptr;
        p.keys = keys + b0;
        p.ticket = ticket;
        p.next_tokens = next_tokens + b0;
        e = launch_lmhead_argmax(p, L);
        if (e != cudaSuccess) return cuda_fail(e, "LM head");
    }
    return A8W8_OK;
}

a8w8_status a8w8_decode_step_i8kv(const a8w8_model* m, const a8w8_config* cfg, int B,
                                  const int32_t* token_ids, const int32_t* slot_mapping,
                                  const int32_t* block_table, int max_blocks, int num_blocks,
                                  const int32_t* ctx_lens, int8_t* const* k_codes,
                                  int8_t* const* v_codes, float* const* k_scales,
                                  float* const* v_scales, const float* rope, int max_pos,
                                  int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                                  void* ws, size_t ws_bytes, void* stream) {
    // the code arrays get the BF16 caches' checks (present, 16-byte aligned)
    a8w8_status s = check_step(m, cfg, B, max_blocks, num_blocks,
                               reinterpret_cast<a8w8_bf16* const*>(k_codes),
                               reinterpret_cast<a8w8_bf16* const*>(v_codes), rope, max_pos,
                               ws_bytes, ws);
    if (s != A8W8_OK) return s;
    if (!k_scales || !v_scales) return fail(A8W8_ERR_INVALID_ARG, "scale arrays are NULL");
    std::vector<KvI8> kv8((size_t)cfg->num_layers);
    for (int l = 0; l < cfg->num_layers; ++l) {
        if ((s = check_ptrs({k_scales[l], v_scales[l]}, "KV row scales")) != A8W8_OK) return s;
        kv8[(size_t)l] = KvI8{k_codes[l], v_codes[l], k_scales[l], v_scales[l]};
    }
    if ((s = check_ptrs({token_ids, slot_mapping, block_table, ctx_lens, next_tokens},
                        "a8w8_decode_step_i8kv")) != A8W8_OK)
        return s;
    if ((logits && !aligned16(logits)) || (final_hidden && !aligned16(final_hidden)))
        return fail(A8W8_ERR_INVALID_ARG, "logits / final_hidden misaligned");
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    return enqueue_step(m, *cfg, B, token_ids, slot_mapping, block_table, max_blocks, num_blocks,
                        ctx_lens, nullptr, nullptr, rope, max_pos, next_tokens, logits,
                        final_hidden, static_cast<unsigned char*>(ws), L, false, kv8.data());
}

a8w8_status a8w8_decode_step(const a8w8_model* m, const a8w8_config* cfg, int B,
                             const int32_t* token_ids, const int32_t* slot_mapping,
                             const int32_t* block_table, int max_blocks, int num_blocks,
                             const int32_t* ctx_lens, a8w8_bf16* const* k_caches,
                             a8w8_bf16* const* v_caches, const float* rope, int max_pos,
                             int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                             void* ws, size_t ws_bytes, void* stream) {
    a8w8_status s = check_step(m, cfg, B, max_blocks, num_blocks, k_caches, v_caches, rope, max_pos,
                               ws_bytes, ws);
    if (s != A8W8_OK) return s;
    if ((s = check_ptrs({token_ids, slot_mapping, block_table, ctx_lens, next_tokens}, "a8w8_decode_step")) != A8W8_OK)
        return s;
    if ((logits && !aligned16(logits)) || (final_hidden && !aligned16(final_hidden)))
        return fail(A8W8_ERR_INVALID_ARG, "logits / final_hidden misaligned");
    Launch L = make_launch(stream, true);
    if (L.num_sms <= 0) return fail(A8W8_ERR_CUDA, "no CUDA device");
    return enqueue_step(m, *cfg, B, token_ids, slot_mapping, block_table, max_blocks, num_blocks,
                        ctx_lens, k_caches, v_caches, rope, max_pos, next_tokens, logits,
                        final_hidden, static_cast<unsigned char*>(ws), L, false);
}

// ---------------------------------------------------------------------------
// Replayable step
// ---------------------------------------------------------------------------

struct a8w8_step_graph {
    int device;
    int B, max_blocks;
    int32_t *tok, *slot, *table, *ctx, *next;
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

static a8w8_status step_graph_create(a8w8_step_graph** out, const a8w8_model* m,
                                     const a8w8_config* cfg, int B, int max_blocks, int num_blocks,
                                     a8w8_bf16* const* k_caches, a8w8_bf16* const* v_caches,
                                     const float* rope, int max_pos, int32_t* token_ids,
                                     int32_t* slot_mapping, int32_t* block_table, int32_t* ctx_lens,
                                     int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                                     int device_loop, void* ws, size_t ws_bytes, void* stream,
                                     const StepSampling* smp) {
    if (!out) return fail(A8W8_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    a8w8_status s = check_step(m, cfg, B, max_blocks, num_blocks, k_caches, v_caches, rope, max_pos,
                               ws_bytes, ws);
    if (s != A8W8_OK) return s;
    if ((s = check_ptrs({token_ids, slot_mapping, block_table, ctx_lens, next_tokens},
                        "a8w8_step_graph_create")) != A8W8_OK)
        return s;
    if ((logits && !aligned16(logits)) || (final_hidden && !aligned16(final_hidden)))
        return fail(A8W8_ERR_INVALID_ARG, "logits / final_hidden misaligned");
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs), "capture status");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(A8W8_ERR_INVALID_ARG, "a8w8_step_graph_create called during stream capture");
    CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize");
    cudaStream_t cap = nullptr;
    CUDA_TRY(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking), "capture stream");
    a8w8_step_graph* g = new a8w8_step_graph();
    cudaGetDevice(&g->device);
    g->B = B;
    g->max_blocks = max_blocks;
    g->tok = token_ids;
    g->slot = slot_mapping;
    g->table = block_table;
    g->ctx = ctx_lens;
    g->next = next_tokens;
    cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        Launch L = make_launch(cap, true);
        s = enqueue_step(m, *cfg, B, g->tok, g->slot, g->table, max_blocks, num_blocks, g->ctx,
                         k_caches, v_caches, rope, max_pos, g->next, logits, final_hidden,
                         static_cast<unsigned char*>(ws), L, device_loop != 0, nullptr, smp);
        cudaGraph_t graph = nullptr;
        cudaError_t e2 = cudaStreamEndCapture(cap, &graph);
        if (s == A8W8_OK && e2 != cudaSuccess) s = cuda_fail(e2, "end capture");
        if (s == A8W8_OK) {
            g->graph = graph;
            e2 = cudaGraphInstantiate(&g->exec, graph, 0);
            if (e2 != cudaSuccess) s = cuda_fail(e2, "graph instantiate");
        } else if (graph) {
            cudaGraphDestroy(graph);
        }
    } else {
        s = cuda_fail(e, "begin capture");
    }
    cudaStreamDestroy(cap);
    if (s != A8W8_OK) {
        if (g->graph) cudaGraphDestroy(g->graph);
        delete g;
        return s;
    }
    *out = g;
    return A8W8_OK;
}

a8w8_status a8w8_step_graph_create(a8w8_step_graph** out, const a8w8_model* m,
                                   const a8w8_config* cfg, int B, int max_blocks, int num_blocks,
                                   a8w8_bf16* const* k_caches, a8w8_bf16* const* v_caches,
                                   const float* rope, int max_pos, int32_t* token_ids,
                                   int32_t* slot_mapping, int32_t* block_table, int32_t* ctx_lens,
                                   int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
                                   int device_loop, void* ws, size_t ws_bytes, void* stream) {
    return step_graph_create(out, m, cfg, B, max_blocks, num_blocks, k_caches, v_caches, rope,
                             max_pos, token_ids, slot_mapping, block_table, ctx_lens, next_tokens,
                             logits, final_hidden, device_loop, ws, ws_bytes, stream, nullptr);
}

a8w8_status a8w8_step_graph_create_sampled(
    a8w8_step_graph** out, const a8w8_model* m, const a8w8_config* cfg, int B, int max_blocks,
    int num_blocks, a8w8_bf16* const* k_caches, a8w8_bf16* const* v_caches, const float* rope,
    int max_pos, int32_t* token_ids, int32_t* slot_mapping, int32_t* block_table,
    int32_t* ctx_lens, int32_t* next_tokens, float* logits, a8w8_bf16* final_hidden,
    int device_loop, float temperature, float top_p, uint64_t seed, uint64_t* step_counter,
    void* sample_ws, size_t sample_ws_bytes, void* ws, size_t ws_bytes, void* stream) {
    if (out) *out = nullptr;
    if (!logits) return fail(A8W8_ERR_INVALID_ARG, "a8w8_step_graph_create_sampled: logits is NULL");
    if (!step_counter || (reinterpret_cast<uintptr_t>(step_counter) & 7))
        return fail(A8W8_ERR_INVALID_ARG, "step_counter NULL or not 8-byte aligned");
    if (!std::isfinite(temperature))
        return fail(A8W8_ERR_INVALID_ARG, "temperature is not finite");
    if (!(top_p > 0.0f && top_p <= 1.0f))
        return fail(A8W8_ERR_INVALID_ARG, "top_p=%g outside (0, 1]", (double)top_p);
    if (cfg && B > 0 && cfg->vocab > 0 &&
        (!sample_ws || !aligned16(sample_ws) || sample_ws_bytes < a8w8_sample_workspace_bytes(B, cfg->vocab)))
        return fail(A8W8_ERR_WORKSPACE, "sampling workspace NULL, misaligned or below %zu bytes",
                    a8w8_sample_workspace_bytes(B, cfg->vocab));
    StepSampling smp;
    smp.T = temperature;
    smp.top_p = top_p;
    smp.seed = seed;
    smp.step = step_counter;
    smp.ws = static_cast<float*>(sample_ws);
    return step_graph_create(out, m, cfg, B, max_blocks, num_blocks, k_caches, v_caches, rope,
                             max_pos, token_ids, slot_mapping, block_table, ctx_lens, next_tokens,
                             logits, final_hidden, device_loop, ws, ws_bytes, stream, &smp);
}

a8w8_status a8w8_step_graph_launch(a8w8_step_graph* g, void* stream) {
    if (!g) return fail(A8W8_ERR_INVALID_ARG, "graph is NULL");
    CUDA_TRY(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)), "graph launch");
    return A8W8_OK;
}

a8w8_status a8w8_step_graph_run_host(a8w8_step_graph* g, const int32_t* token_ids,
                                     const int32_t* slot_mapping, const int32_t* block_table,
                                     const int32_t* ctx_lens, int32_t* next_tokens, void* stream) {
    if (!g) return fail(A8W8_ERR_INVALID_ARG, "graph is NULL");
    if (!token_ids || !slot_mapping || !block_table || !ctx_lens || !next_tokens)
        return fail(A8W8_ERR_INVALID_ARG, "a8w8_step_graph_run_host: NULL host buffer");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t b4 = (size_t)g->B * sizeof(int32_t);
    CUDA_TRY(cudaMemcpyAsync(g->tok, token_ids, b4, cudaMemcpyHostToDevice, st), "H2D tokens");
    CUDA_TRY(cudaMemcpyAsync(g->slot, slot_mapping, b4, cudaMemcpyHostToDevice, st), "H2D slots");
    CUDA_TRY(cudaMemcpyAsync(g->table, block_table, b4 * g->max_blocks, cudaMemcpyHostToDevice, st),
             "H2D block table");
    CUDA_TRY(cudaMemcpyAsync(g->ctx, ctx_lens, b4, cudaMemcpyHostToDevice, st), "H2D ctx lens");
    CUDA_TRY(cudaGraphLaunch(g->exec, st), "graph launch");
    CUDA_TRY(cudaMemcpyAsync(next_tokens, g->next, b4, cudaMemcpyDeviceToHost, st), "D2H next tokens");
    CUDA_TRY(cudaStreamSynchronize(st), "stream synchronize");
    return A8W8_OK;
}

void a8w8_step_graph_destroy(a8w8_step_graph* g) {
    if (!g) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(g->device);
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    cudaSetDevice(cur);
    delete g;
}

}  // extern "C"
