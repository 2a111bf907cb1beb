// attn_i8.cu -- the INT8 KV cache variant: K/V rows stored as INT8 codes with
// one FP32 scale per (token, KV head) row, quantised when written and
// dequantised where attention reads them.
//
// "perf(qwen3-a8w8): optimize decode scheduling and data paths" (pypto-lib PR
// #810), "BF16 KV cache", names the storage that BF16 replaced: INT8 K/V cache
// rows plus FP32 row scales, per-token K/V quantisation in decode and prefill,
// per-row dequantisation inside attention, the scales in tensors of their own.
// A row is one KV head's D values of one token; it is quantised with the
// activation formula (s = absmax / 127, q = clamp(rne(x / s), -127, 127), IEEE
// float32 quotients) from the BF16 values the BF16 cache would hold.
//
// Attention follows the per-head BF16 form of attn_impl.cuh step for step,
// with two changes that keep its two-float accuracy:
//   * score_t = ((sum_d q_d c_d) * s_t) * scale: each q_d c_d (a BF16 value
//     times an integer of at most 7 bits) is exact in float32 and the sum is a
//     two-float pair, multiplied by the row scale s_t as a pair;
//   * o_d = sum_t (p_t * sv_t) * c_d: the probability pair times the V row's
//     scale, then times the code; the denominator l sums p_t alone.
// K/V tiles hold the codes (1 byte per element instead of 2) and the row
// scales. Partials and the combine are those of the BF16 form.
#include "attn_impl.cuh"

namespace a8w8 {

namespace {

constexpr int kI8TilePad = 16;   // code tile rows of D + 16 bytes (16-byte aligned)

// Shared memory of one item: K and V code tiles, then the K and V row scales
// (after P.V the region holds the in-kernel combine's scratch), the query row
// (float), scores (hi and lo planes), (m, l), the flag and the maximum's key.
__host__ __device__ inline size_t i8_tiles_bytes(int chunk, int D) {
    const size_t kv = (size_t)2 * chunk * (D + kI8TilePad) + (size_t)2 * chunk * 4;
    const size_t comb = (size_t)(2 * kMaxInKernelSplits + 2) * 4 + (size_t)(kMaxInKernelSplits + 1) * 4;
    return kv > comb ? kv : comb;
}
__host__ __device__ inline size_t i8_item_smem_bytes(int chunk, int D) {
    return i8_tiles_bytes(chunk, D) + (size_t)D * 4 + (size_t)2 * chunk * 4 + 4 * 4 + 16;
}

// Row quantisation of the lane's E = D / 32 elements of one head row held by
// a warp: the row scale (identical on every lane) and the codes.
template <int E>
__device__ __forceinline__ float quant_row_warp(const float (&x)[E], int (&c)[E]) {
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
    amax = warp_max(amax);
    const float sc = __fdiv_rn(amax, 127.0f);
    const float rc = quant_recip(sc);
#pragma unroll
    for (int e = 0; e < E; ++e) c[e] = quant_code(x[e], sc, rc);
    return sc;
}

// One attention work item (request b, query head h, token chunk `split`) on
// the first NT threads of the CTA; same structure and synchronisation as
// attn_item in attn_impl.cuh.
template <int D, int NT>
__device__ __forceinline__ void attn_i8_item(const AttnI8Params& P, int chunk, int splits,
                                             int split, int h, int b, unsigned char* smem) {
    const AttnParams& p = P.a;
    constexpr int NW = NT / 32;
    constexpr int DP = D + kI8TilePad;
    static_assert(D % 32 == 0 && DP % 16 == 0, "16-byte code rows and tile pitch");
    int8_t* Ks = reinterpret_cast<int8_t*>(smem);
    int8_t* Vs = Ks + (size_t)chunk * DP;
    float* kss = reinterpret_cast<float*>(Vs + (size_t)chunk * DP);   // [chunk]
    float* vss = kss + chunk;                                         // [chunk]
    float* qs = reinterpret_cast<float*>(smem + i8_tiles_bytes(chunk, D));   // [D]
    float* sc = qs + D;                            // [chunk] hi
    float* sl = sc + chunk;                        // [chunk] lo
    float* stat = sl + chunk;                      // m hi, m lo, l hi, l lo
    int* s_flag = reinterpret_cast<int*>(stat + 4);
    unsigned long long* s_mkey = reinterpret_cast<unsigned long long*>(stat + 6);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = p.Hq / p.Hkv;
    const int kvh = h / G;
    const bool lead = h - kvh * G == 0;            // the head that writes the new K/V
    const int t0 = split * chunk;
    const int max_ctx = p.max_blocks * p.page;
    const int ctx_raw = p.ctx_lens[b];
    const bool bad_ctx = ctx_raw < 0 || ctx_raw > max_ctx;
    const int pos = ctx_raw - 1;
    const bool bad_pos = p.fused && !bad_ctx && ctx_raw > 0 && pos >= p.max_pos;
    const int ctx = (bad_ctx || bad_pos) ? 0 : ctx_raw;
    const int t1 = min(t0 + chunk, ctx);
    const int n = max(t1 - t0, 0);
    const bool covers_new = p.fused && ctx > 0 && pos >= t0 && pos < t0 + chunk;
    const int n_old = covers_new ? n - 1 : n;
    const int active = p.tickets ? max(1, (ctx + chunk - 1) / chunk) : splits;
    if (split >= active) return;   // the whole CTA, before any barrier
    const bool single = active == 1;

    if (tid == 0) {
        *s_flag = 0;
        *s_mkey = 0ull;
    }
    attn_sync<NT>();
    // cached rows: codes by 16-byte copies, row scales by plain loads
    constexpr int RV = D / 16;
    for (int i = tid; i < n_old * RV; i += NT) {
        const int t = i / RV, c = i - t * RV;
        const int tok = t0 + t;
        const int blk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        if (blk < 0 || blk >= p.num_blocks) {
            *reinterpret_cast<int4*>(Ks + (size_t)t * DP + 16 * c) = make_int4(0, 0, 0, 0);
            *reinterpret_cast<int4*>(Vs + (size_t)t * DP + 16 * c) = make_int4(0, 0, 0, 0);
            *s_flag = 1;
            continue;
        }
        const size_t row = ((size_t)blk * p.page + tok % p.page) * p.Hkv + kvh;
        cp_async16(Ks + (size_t)t * DP + 16 * c, P.k_codes + row * D + 16 * c);
        cp_async16(Vs + (size_t)t * DP + 16 * c, P.v_codes + row * D + 16 * c);
    }
    cp_async_commit();
    for (int t = tid; t < n_old; t += NT) {
        const int tok = t0 + t;
        const int blk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        float ks = 0.0f, vs = 0.0f;
        if (blk >= 0 && blk < p.num_blocks) {
            const size_t row = ((size_t)blk * p.page + tok % p.page) * p.Hkv + kvh;
            ks = __ldcg(P.k_scale + row);
            vs = __ldcg(P.v_scale + row);
        }
        kss[t] = ks;
        vss[t] = vs;
    }
    HeadPre<D> hp;
    if (p.fused && n > 0 && warp < 2) load_head_pre<D>(p, pos < p.max_pos ? pos : 0, lane, hp);

    pdl_wait();
    pdl_trigger();

    if (tid == 0) {
        if (bad_ctx) set_error(p.err, 0x4u);
        if (bad_pos) set_error(p.err, 0x10u);
    }

    // warp 0: the query head; warp 1: the new token's K (norm + RoPE) and V,
    // quantised per row into the tiles and, by the group's lead head, the cache
    constexpr int E = D / 32;
    if (n > 0 && warp == 0) {
        const bf16* src = p.q + (size_t)b * p.q_stride + (size_t)h * D;
        float x[E], y[E];
        load_bf16_lane<D>(src + lane * E, x);
        if (p.fused) {
            norm_rope_head<D>(x, hp.qw, hp, p.eps, lane, y);
            if (p.tap_q_rot && split == 0) {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    p.tap_q_rot[((size_t)b * p.Hq + h) * D + lane * E + e] = f2bf(y[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) y[e] = x[e];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) qs[lane * E + e] = y[e];
    } else if (n > 0 && warp == 1 && covers_new) {
        const int NQ = p.Hq * D, NK = p.Hkv * D;
        const bf16* ksrc = p.q + (size_t)b * p.q_stride + NQ + (size_t)kvh * D;
        const bf16* vsrc = p.q + (size_t)b * p.q_stride + NQ + NK + (size_t)kvh * D;
        float x[E], vv[E], y[E];
        load_bf16_lane<D>(ksrc + lane * E, x);
        load_bf16_lane<D>(vsrc + lane * E, vv);
        norm_rope_head<D>(x, hp.kw, hp, p.eps, lane, y);
        int kc[E], vc[E];
        const float ks = quant_row_warp<E>(y, kc);
        const float vs = quant_row_warp<E>(vv, vc);
        const int tr = pos - t0;
        const long slot = p.slot_mapping[b];
        const long num_slots = (long)p.num_blocks * p.page;
        const bool slot_ok = lead && slot >= 0 && slot < num_slots;
        if (lead && lane == 0 && slot >= num_slots) set_error(p.err, 0x1u);
        if (lane == 0) {
            kss[tr] = ks;
            vss[tr] = vs;
            if (slot_ok) {
                P.k_scale[(size_t)slot * p.Hkv + kvh] = ks;
                P.v_scale[(size_t)slot * p.Hkv + kvh] = vs;
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            Ks[(size_t)tr * DP + d] = (int8_t)kc[e];
            Vs[(size_t)tr * DP + d] = (int8_t)vc[e];
            if (slot_ok) {
                P.k_codes[((size_t)slot * p.Hkv + kvh) * D + d] = (int8_t)kc[e];
                P.v_codes[((size_t)slot * p.Hkv + kvh) * D + d] = (int8_t)vc[e];
            }
            if (lead && p.tap_k_rot) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = f2bf(y[e]);
        }
    }
    cp_async_wait_all();
    attn_sync<NT>();
    if (tid == 0 && *s_flag) set_error(p.err, 0x2u);

    // scores: one token per LPT lanes, 8 codes per lane
    constexpr int LPT = D / 8;
    constexpr int PPW = 32 / LPT;
    const f2 scale = {p.scale, p.scale_lo};
    {
        const int j = lane % LPT, pw = lane / LPT;
        const float4 qa = *reinterpret_cast<const float4*>(qs + 8 * j);
        const float4 qb = *reinterpret_cast<const float4*>(qs + 8 * j + 4);
        const int step = NW * PPW;
        const int n_pad = (n + step - 1) / step * step;
        for (int t = warp * PPW + pw; t < n_pad; t += step) {
            const bool ok = t < n;
            const uint2 raw = *reinterpret_cast<const uint2*>(Ks + (size_t)(ok ? t : 0) * DP + 8 * j);
            const char4 c0 = *reinterpret_cast<const char4*>(&raw.x);
            const char4 c1 = *reinterpret_cast<const char4*>(&raw.y);
            f2 d = f2_make(__fmul_rn(qa.x, (float)c0.x));
            f2_acc(d, __fmul_rn(qa.y, (float)c0.y));
            f2_acc(d, __fmul_rn(qa.z, (float)c0.z));
            f2_acc(d, __fmul_rn(qa.w, (float)c0.w));
            f2_acc(d, __fmul_rn(qb.x, (float)c1.x));
            f2_acc(d, __fmul_rn(qb.y, (float)c1.y));
            f2_acc(d, __fmul_rn(qb.z, (float)c1.z));
            f2_acc(d, __fmul_rn(qb.w, (float)c1.w));
#pragma unroll
            for (int o = LPT / 2; o > 0; o >>= 1) {
                f2 r;
                r.hi = __shfl_xor_sync(0xffffffffu, d.hi, o);
                r.lo = __shfl_xor_sync(0xffffffffu, d.lo, o);
                d = f2_add(d, r);
            }
            if (j == 0 && ok) {
                const f2 sv = f2_mul(f2_mulf(d, kss[t]), scale);
                sc[t] = sv.hi;
                sl[t] = sv.lo;
                atomicMax(s_mkey, f2_key(sv));
            }
        }
    }
    attn_sync<NT>();

    // softmax numerators p_t = exp(s_t - m), one token per thread
    {
        const unsigned long long mk = *s_mkey;
        const f2 m = {unord32((unsigned)(mk >> 32)), unord32((unsigned)mk)};
        if (tid == 0) {
            stat[0] = m.hi;
            stat[1] = m.lo;
        }
        for (int t = tid; t < n; t += NT) {
            const f2 e = f2_exp(f2_sub(f2{sc[t], sl[t]}, m));
            sc[t] = e.hi;
            sl[t] = e.lo;
        }
    }
    attn_sync<NT>();

    // P.V: TG consecutive lanes share a column pair and split the tokens
    {
        constexpr int CP = D / 2;
        constexpr int TG = NT / CP;
        static_assert(TG >= 1 && TG <= 32 && (TG & (TG - 1)) == 0, "token groups");
        const int cp = tid / TG, tg = tid % TG;
        f2 o0 = {0.0f, 0.0f}, o1 = {0.0f, 0.0f}, l = {0.0f, 0.0f};
        for (int t = tg; t < n; t += TG) {
            const char2 v = *reinterpret_cast<const char2*>(Vs + (size_t)t * DP + 2 * cp);
            const f2 pr = {sc[t], sl[t]};
            const f2 pv = f2_mulf(pr, vss[t]);
            o0 = f2_add(o0, f2_mulf(pv, (float)v.x));
            o1 = f2_add(o1, f2_mulf(pv, (float)v.y));
            l = f2_add(l, pr);
        }
#pragma unroll
        for (int o = TG / 2; o > 0; o >>= 1) {
            f2 r;
            r.hi = __shfl_xor_sync(0xffffffffu, o0.hi, o);
            r.lo = __shfl_xor_sync(0xffffffffu, o0.lo, o);
            o0 = f2_add(o0, r);
            r.hi = __shfl_xor_sync(0xffffffffu, o1.hi, o);
            r.lo = __shfl_xor_sync(0xffffffffu, o1.lo, o);
            o1 = f2_add(o1, r);
            r.hi = __shfl_xor_sync(0xffffffffu, l.hi, o);
            r.lo = __shfl_xor_sync(0xffffffffu, l.lo, o);
            l = f2_add(l, r);
        }
        if (tg == 0) {
            if (single) {
                bf16* out = p.out + ((size_t)b * p.Hq + h) * D + 2 * cp;
                out[0] = n > 0 ? f2_to_bf16(f2_div(o0, l)) : __float2bfloat16_rn(0.0f);
                out[1] = n > 0 ? f2_to_bf16(f2_div(o1, l)) : __float2bfloat16_rn(0.0f);
            } else {
                float* pp = p.part + (((size_t)b * p.Hq + h) * splits + split) * (2 * D + 4);
                pp[2 * cp] = n > 0 ? o0.hi : 0.0f;
                pp[2 * cp + 1] = n > 0 ? o1.hi : 0.0f;
                pp[D + 2 * cp] = n > 0 ? o0.lo : 0.0f;
                pp[D + 2 * cp + 1] = n > 0 ? o1.lo : 0.0f;
                if (cp == 0) {
                    pp[2 * D] = n > 0 ? stat[0] : -INFINITY;
                    pp[2 * D + 1] = n > 0 ? stat[1] : 0.0f;
                    pp[2 * D + 2] = n > 0 ? l.hi : 0.0f;
                    pp[2 * D + 3] = n > 0 ? l.lo : 0.0f;
                }
            }
        }
    }
    if (!single && p.tickets) {
        // the last CTA of this (request, query head) combines the partials
        __threadfence();
        attn_sync<NT>();
        if (tid == 0) {
            unsigned* tk = p.tickets + (size_t)b * p.Hq + h;
            const unsigned prev = atomicAdd(tk, 1u);
            *s_flag = prev == (unsigned)(active - 1);
            if (*s_flag) *tk = 0u;
        }
        attn_sync<NT>();
        if (*s_flag) {
            __threadfence();
            float* cw = reinterpret_cast<float*>(smem);            // [splits][2]
            float* cl = cw + 2 * kMaxInKernelSplits;               // [2]
            int* act = reinterpret_cast<int*>(cl + 2);             // [splits]
            int* nact = act + kMaxInKernelSplits;                  // [1]
            const float* pb = p.part + ((size_t)b * p.Hq + h) * splits * (2 * D + 4);
            if (warp == 0) combine_weights<D>(pb, active, cw, cl, lane, act, nact);
            attn_sync<NT>();
            for (int d = tid; d < D; d += NT) {
                f2 acc = {0.0f, 0.0f};
                for (int k = 0; k < *nact; ++k) {
                    const int sp = act[k];
                    const float* q = pb + (size_t)sp * (2 * D + 4);
                    acc = f2_add(acc, f2_mul(f2{__ldcg(q + d), __ldcg(q + D + d)},
                                             f2{cw[2 * sp], cw[2 * sp + 1]}));
                }
                const f2 l = {cl[0], cl[1]};
                p.out[((size_t)b * p.Hq + h) * D + d] =
                    l.hi > 0.0f ? f2_to_bf16(f2_div(acc, l)) : __float2bfloat16_rn(0.0f);
            }
        }
    }
    attn_sync<NT>();
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_i8_kernel(const AttnI8Params P, int chunk,
                                                               int splits) {
    extern __shared__ __align__(16) unsigned char smem[];
    attn_i8_item<D, kAttnThreads>(P, chunk, splits, blockIdx.x, blockIdx.y, blockIdx.z, smem);
}

// Separate combine of the standalone entry: one CTA per (query head, request).
template <int D>
__global__ void __launch_bounds__(D) attn_i8_combine_kernel(const float* __restrict__ part,
                                                            int splits, int Hq,
                                                            bf16* __restrict__ out) {
    extern __shared__ float cws[];   // [splits][2] weights, then L[2]
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y;
    const float* pp = part + ((size_t)b * Hq + h) * splits * (2 * D + 4);
    if (threadIdx.x < 32) combine_weights<D>(pp, splits, cws, cws + 2 * splits, threadIdx.x);
    __syncthreads();
    out[((size_t)b * Hq + h) * D + threadIdx.x] =
        combine_elem<D>(pp, splits, cws, cws + 2 * splits, threadIdx.x);
}

// Quantise-on-write of k, v [T, Hkv, D] into the INT8 cache: one warp per
// (token, KV head) row, E = D / 32 elements per lane.
template <int D>
__global__ void __launch_bounds__(256) kv_write_i8_kernel(const bf16* __restrict__ k,
                                                          const bf16* __restrict__ v, int T,
                                                          int Hkv,
                                                          const int32_t* __restrict__ slot_mapping,
                                                          int8_t* __restrict__ k_codes,
                                                          int8_t* __restrict__ v_codes,
                                                          float* __restrict__ k_scale,
                                                          float* __restrict__ v_scale,
                                                          long num_slots, unsigned* err) {
    constexpr int E = D / 32;
    static_assert(D % 32 == 0, "whole lanes per row");
    pdl_wait();
    pdl_trigger();
    const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);   // token * Hkv + head
    const int lane = threadIdx.x & 31;
    if (row >= (long)T * Hkv) return;                            // whole warps
    const int t = (int)(row / Hkv), hh = (int)(row - (long)t * Hkv);
    const long slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && hh == 0) set_error(err, 0x1u);
        return;
    }
    float x[E], y[E];
    load_bf16_lane<D>(k + (size_t)row * D + lane * E, x);
    load_bf16_lane<D>(v + (size_t)row * D + lane * E, y);
    int kc[E], vc[E];
    const float ks = quant_row_warp<E>(x, kc);
    const float vs = quant_row_warp<E>(y, vc);
    const size_t dst = ((size_t)slot * Hkv + hh) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        k_codes[dst + e] = (int8_t)kc[e];
        v_codes[dst + e] = (int8_t)vc[e];
    }
    if (lane == 0) {
        k_scale[(size_t)slot * Hkv + hh] = ks;
        v_scale[(size_t)slot * Hkv + hh] = vs;
    }
}

// ---------------------------------------------------------------------------
// Grouped form (large batches, long contexts): one CTA per (request, KV head,
// 128-token chunk) for every query head of the group, as attn_group.cu does for
// the BF16 cache, over code tiles. Both row-scale arrays are read with the
// block ids; the softmax stores p_t * v_scale_t (a pair product) for P.V while
// the denominator l sums p_t alone, so P.V multiplies those pairs by the codes.
// Decode only (the new token is quantised here, not by a prefill pre-pass).
// ---------------------------------------------------------------------------
constexpr int kG8Threads = 256;
constexpr int kG8Chunk = 128;        // the BF16 grouped form's chunk ...
constexpr int kG8MaxG = 7;           // ... heads per KV head ...
constexpr int kG8MaxSplits = 64;     // ... and chunks per request (attn_group_shape_ok)

__host__ __device__ inline size_t al16(size_t x) { return (x + 15) & ~size_t(15); }

struct G8Smem {
    size_t tile, vnew, ksc, vsc, q, pr, stat, blk, flag, total;
};
__host__ __device__ inline G8Smem g8_smem(int D, int G) {
    G8Smem s;
    s.tile = 0;
    const size_t kv = (size_t)kG8Chunk * (D + kI8TilePad);
    // combine scratch reuses the tile: per head 2*splits weights, 2 for L,
    // splits active indices and their count
    const size_t comb = (size_t)G * (2 * kG8MaxSplits + 2 + kG8MaxSplits + 1) * 4;
    s.vnew = al16(kv > comb ? kv : comb);                // [D] int8: the new token's V codes
    s.ksc = s.vnew + al16((size_t)D);                    // [chunk] K row scales
    s.vsc = s.ksc + (size_t)kG8Chunk * 4;                // [chunk] V row scales
    s.q = s.vsc + (size_t)kG8Chunk * 4;                  // [G][D] float
    s.pr = s.q + (size_t)G * D * 4;                      // [G][chunk] (hi, lo) pairs
    s.stat = s.pr + (size_t)G * kG8Chunk * 8;            // [G][4]: m hi, m lo, l hi, l lo
    s.blk = s.stat + (size_t)G * 4 * 4;                  // [chunk] physical block per token
    s.flag = s.blk + (size_t)kG8Chunk * 4;
    s.total = s.flag + 16;
    return s;
}

// acc += p * v with p a pair and v a float (Dot2 accumulation: the product's
// high part by TwoSum, the rounding errors into acc.lo).
__device__ __forceinline__ void dot2_acc8(f2& acc, const f2 p, float v) {
    const float h = __fmul_rn(p.hi, v);
    const float e = __fmaf_rn(p.hi, v, -h);
    float s, err;
    two_sum(acc.hi, h, s, err);
    acc.hi = s;
    acc.lo = __fadd_rn(acc.lo, __fadd_rn(err, __fmaf_rn(p.lo, v, e)));
}

template <int D, int G>
__global__ void __launch_bounds__(kG8Threads) attn_i8_group_kernel(const AttnI8Params P, int splits) {
    static_assert(G >= 1 && G <= kG8MaxG, "query heads per KV head");
    static_assert(D % 32 == 0 && (D + kI8TilePad) % 16 == 0, "16-byte code rows and tile pitch");
    const AttnParams& p = P.a;
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NT = kG8Threads, C = kG8Chunk;
    constexpr int DP = D + kI8TilePad;
    constexpr int RV = D / 16;        // 16-byte code vectors per row
    constexpr int E = D / 32;
    const G8Smem L = g8_smem(D, G);
    int8_t* Ts = reinterpret_cast<int8_t*>(smem + L.tile);   // K codes, then V codes
    int8_t* vnew = reinterpret_cast<int8_t*>(smem + L.vnew);
    float* ksc = reinterpret_cast<float*>(smem + L.ksc);
    float* vsc = reinterpret_cast<float*>(smem + L.vsc);
    float* qs = reinterpret_cast<float*>(smem + L.q);
    float2* pr = reinterpret_cast<float2*>(smem + L.pr);
    float* stat = reinterpret_cast<float*>(smem + L.stat);
    int* blk = reinterpret_cast<int*>(smem + L.blk);
    int* s_flag = reinterpret_cast<int*>(smem + L.flag);

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = kvh * G;
    const int t0 = split * C;
    const int max_ctx = p.max_blocks * p.page;
    const int ctx_raw = p.ctx_lens[b];
    const bool bad_ctx = ctx_raw < 0 || ctx_raw > max_ctx;
    const int pos = ctx_raw - 1;
    const bool bad_pos = !bad_ctx && ctx_raw > 0 && pos >= p.max_pos;
    const int ctx = (bad_ctx || bad_pos) ? 0 : ctx_raw;
    const int n = max(min(t0 + C, ctx) - t0, 0);
    const bool covers_new = ctx > 0 && pos >= t0 && pos < t0 + C;
    const int n_old = covers_new ? n - 1 : n;
    const int active = max(1, (ctx + C - 1) / C);
    if (split >= active) return;   // the whole CTA, before any barrier
    const bool single = active == 1;

    // physical block and row scales of every cached token of the chunk
    // (prefill: the scales and codes of this launch's tokens are written by the
    // pre-pass before, so they are read only after the dependency wait)
    if (p.kv_in_cache) pdl_wait();
    if (tid == 0) *s_flag = 0;
    for (int t = tid; t < n_old; t += NT) {
        const int tok = t0 + t;
        const int bk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        const bool ok = bk >= 0 && bk < p.num_blocks;
        blk[t] = ok ? bk : -1;
        float ks = 0.0f, vs = 0.0f;
        if (ok) {
            const size_t row = ((size_t)bk * p.page + tok % p.page) * p.Hkv + kvh;
            ks = __ldcg(P.k_scale + row);
            vs = __ldcg(P.v_scale + row);
        }
        ksc[t] = ks;
        vsc[t] = vs;
    }
    __syncthreads();
    // code rows of the cached tokens of `cache` into the tile (zeros for a bad block)
    auto load_tile = [&](const int8_t* cache) {
        for (int i = tid; i < n_old * RV; i += NT) {
            const int t = i / RV, c = i - t * RV;
            const int bk = blk[t];
            if (bk < 0) {
                *reinterpret_cast<int4*>(Ts + (size_t)t * DP + 16 * c) = make_int4(0, 0, 0, 0);
                *s_flag = 1;
                continue;
            }
            const int tok = t0 + t;
            const size_t off = (((size_t)bk * p.page + tok % p.page) * p.Hkv + kvh) * D + 16 * c;
            cp_async16(Ts + (size_t)t * DP + 16 * c, cache + off);
        }
        cp_async_commit();
    };
    load_tile(P.k_codes);
    // warps 0..G-1: query heads; warp G: the new token's K and V
    const bool qwarp = warp < G;
    const bool kwarp = warp == G && covers_new;
    HeadPre<D> hp;
    if (n > 0 && (qwarp || kwarp)) load_head_pre<D>(p, pos < p.max_pos ? pos : 0, lane, hp);

    pdl_wait();
    pdl_trigger();

    if (tid == 0) {
        if (bad_ctx) set_error(p.err, 0x4u);
        if (bad_pos) set_error(p.err, 0x10u);
    }
    if (n > 0 && qwarp) {
        const int h = h0 + warp;
        float x[E], y[E];
        load_bf16_lane<D>(p.q + (size_t)b * p.q_stride + (size_t)h * D + lane * E, x);
        norm_rope_head<D>(x, hp.qw, hp, p.eps, lane, y);
#pragma unroll
        for (int e = 0; e < E; ++e) qs[warp * D + lane * E + e] = y[e];
        if (p.tap_q_rot && split == 0) {
#pragma unroll
            for (int e = 0; e < E; ++e)
                p.tap_q_rot[((size_t)b * p.Hq + h) * D + lane * E + e] = f2bf(y[e]);
        }
    } else if (n > 0 && kwarp) {
        const int NQ = p.Hq * D, NK = p.Hkv * D;
        const bf16* row = p.q + (size_t)b * p.q_stride;
        float x[E], vv[E], y[E];
        load_bf16_lane<D>(row + NQ + (size_t)kvh * D + lane * E, x);
        load_bf16_lane<D>(row + NQ + NK + (size_t)kvh * D + lane * E, vv);
        norm_rope_head<D>(x, hp.kw, hp, p.eps, lane, y);
        int kc[E], vc[E];
        const float ks = quant_row_warp<E>(y, kc);
        const float vs = quant_row_warp<E>(vv, vc);
        const int tr = pos - t0;
        const long slot = p.slot_mapping[b];
        const long num_slots = (long)p.num_blocks * p.page;
        // prefill: the pre-pass has written the cache (and flagged a bad slot)
        const bool write = !p.kv_in_cache;
        const bool slot_ok = write && slot >= 0 && slot < num_slots;
        if (lane == 0) {
            if (write && slot >= num_slots) set_error(p.err, 0x1u);
            ksc[tr] = ks;
            vsc[tr] = vs;
            if (slot_ok) {
                P.k_scale[(size_t)slot * p.Hkv + kvh] = ks;
                P.v_scale[(size_t)slot * p.Hkv + kvh] = vs;
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            Ts[(size_t)tr * DP + d] = (int8_t)kc[e];
            vnew[d] = (int8_t)vc[e];
            if (slot_ok) {
                P.k_codes[((size_t)slot * p.Hkv + kvh) * D + d] = (int8_t)kc[e];
                P.v_codes[((size_t)slot * p.Hkv + kvh) * D + d] = (int8_t)vc[e];
            }
            if (p.tap_k_rot && write) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = f2bf(y[e]);
        }
    }
    cp_async_wait_all();
    __syncthreads();
    if (tid == 0 && *s_flag) set_error(p.err, 0x2u);

    // scores: warp w takes tokens 32 (w % 4) + lane and heads w / 4, +2, +4, +6
    const f2 scale = {p.scale, p.scale_lo};
    {
        const int t = (warp & 3) * 32 + lane;
        const int hb = warp >> 2;
        constexpr int HW = (G + 1) / 2;    // heads per warp, at most
        if (t < n) {
            f2 acc[HW];
#pragma unroll
            for (int i = 0; i < HW; ++i) acc[i] = f2{0.0f, 0.0f};
            const int8_t* krow = Ts + (size_t)t * DP;
#pragma unroll 2
            for (int dv = 0; dv < D / 8; ++dv) {
                const uint2 raw = *reinterpret_cast<const uint2*>(krow + 8 * dv);
                const char4 c0 = *reinterpret_cast<const char4*>(&raw.x);
                const char4 c1 = *reinterpret_cast<const char4*>(&raw.y);
                const float kf[8] = {(float)c0.x, (float)c0.y, (float)c0.z, (float)c0.w,
                                     (float)c1.x, (float)c1.y, (float)c1.z, (float)c1.w};
#pragma unroll
                for (int i = 0; i < HW; ++i) {
                    const int hh = hb + 2 * i;
                    if (hh < G) {
                        const float4 qa = *reinterpret_cast<const float4*>(qs + hh * D + 8 * dv);
                        const float4 qb = *reinterpret_cast<const float4*>(qs + hh * D + 8 * dv + 4);
                        f2_acc(acc[i], __fmul_rn(qa.x, kf[0]));
                        f2_acc(acc[i], __fmul_rn(qa.y, kf[1]));
                        f2_acc(acc[i], __fmul_rn(qa.z, kf[2]));
                        f2_acc(acc[i], __fmul_rn(qa.w, kf[3]));
                        f2_acc(acc[i], __fmul_rn(qb.x, kf[4]));
                        f2_acc(acc[i], __fmul_rn(qb.y, kf[5]));
                        f2_acc(acc[i], __fmul_rn(qb.z, kf[6]));
                        f2_acc(acc[i], __fmul_rn(qb.w, kf[7]));
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < HW; ++i) {
                const int hh = hb + 2 * i;
                if (hh < G) {
                    const f2 d = f2_mulf(fast_two_sum(acc[i].hi, acc[i].lo), ksc[t]);
                    const f2 sv = f2_mul(d, scale);
                    pr[hh * C + t] = make_float2(sv.hi, sv.lo);
                }
            }
        }
    }
    __syncthreads();   // the K tile is no longer read

    // the V codes into the same buffer, behind the softmax
    load_tile(P.v_codes);
    if (n > 0 && warp == G && covers_new) {
        for (int d = lane; d < D; d += 32) Ts[(size_t)(pos - t0) * DP + d] = vnew[d];
    }

    // softmax of head w over the chunk: p = exp(s - m), l = sum p; the pairs
    // kept for P.V are p * v_scale
    if (warp < G) {
        float2* ph = pr + warp * C;
        f2 m = {-INFINITY, 0.0f};
        for (int t = lane; t < n; t += 32) m = f2_max(m, f2{ph[t].x, ph[t].y});
        m = warp_max_f2(m);
        f2 l = {0.0f, 0.0f};
        for (int t = lane; t < n; t += 32) {
            const f2 e = f2_exp(f2_sub(f2{ph[t].x, ph[t].y}, m));
            l = f2_add(l, e);
            const f2 w = f2_mulf(e, vsc[t]);
            ph[t] = make_float2(w.hi, w.lo);
        }
        l = warp_sum_f2(l);
        if (lane == 0) {
            stat[warp * 4 + 0] = m.hi;
            stat[warp * 4 + 1] = m.lo;
            stat[warp * 4 + 2] = l.hi;
            stat[warp * 4 + 3] = l.lo;
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // P.V: TG consecutive threads share a column pair and split the tokens
    {
        constexpr int CP = D / 2;
        constexpr int TG = NT / CP;
        static_assert(TG >= 1 && TG <= 32 && (TG & (TG - 1)) == 0, "token groups");
        const int cp = tid / TG, tg = tid % TG;
        f2 o[G][2];
#pragma unroll
        for (int h = 0; h < G; ++h) o[h][0] = o[h][1] = f2{0.0f, 0.0f};
        for (int t = tg; t < n; t += TG) {
            const char2 v = *reinterpret_cast<const char2*>(Ts + (size_t)t * DP + 2 * cp);
            const float v0 = (float)v.x, v1 = (float)v.y;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 q = pr[h * C + t];
                dot2_acc8(o[h][0], f2{q.x, q.y}, v0);
                dot2_acc8(o[h][1], f2{q.x, q.y}, v1);
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            o[h][0] = fast_two_sum(o[h][0].hi, o[h][0].lo);
            o[h][1] = fast_two_sum(o[h][1].hi, o[h][1].lo);
#pragma unroll
            for (int s = TG / 2; s > 0; s >>= 1) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    f2 r;
                    r.hi = __shfl_xor_sync(0xffffffffu, o[h][c].hi, s);
                    r.lo = __shfl_xor_sync(0xffffffffu, o[h][c].lo, s);
                    o[h][c] = f2_add(o[h][c], r);
                }
            }
        }
        if (tg == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const int hq = h0 + h;
                const f2 l = {stat[h * 4 + 2], stat[h * 4 + 3]};
                if (single) {
                    bf16* out = p.out + ((size_t)b * p.Hq + hq) * D + 2 * cp;
                    out[0] = n > 0 ? f2_to_bf16(f2_div(o[h][0], l)) : __float2bfloat16_rn(0.0f);
                    out[1] = n > 0 ? f2_to_bf16(f2_div(o[h][1], l)) : __float2bfloat16_rn(0.0f);
                } else {
                    float* pp = p.part + (((size_t)b * p.Hq + hq) * splits + split) * (2 * D + 4);
                    pp[2 * cp] = n > 0 ? o[h][0].hi : 0.0f;
                    pp[2 * cp + 1] = n > 0 ? o[h][1].hi : 0.0f;
                    pp[D + 2 * cp] = n > 0 ? o[h][0].lo : 0.0f;
                    pp[D + 2 * cp + 1] = n > 0 ? o[h][1].lo : 0.0f;
                    if (cp == 0) {
                        pp[2 * D] = n > 0 ? stat[h * 4 + 0] : -INFINITY;
                        pp[2 * D + 1] = n > 0 ? stat[h * 4 + 1] : 0.0f;
                        pp[2 * D + 2] = n > 0 ? l.hi : 0.0f;
                        pp[2 * D + 3] = n > 0 ? l.lo : 0.0f;
                    }
                }
            }
        }
    }
    if (single) return;   // no barrier follows on this path

    // the last CTA of this (request, KV head) merges the chunks' partials
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        unsigned* tk = p.tickets + (size_t)b * p.Hq + kvh;
        const unsigned prev = atomicAdd(tk, 1u);
        *s_flag = prev == (unsigned)(active - 1);
        if (*s_flag) *tk = 0u;   // ready for the next launch
    }
    __syncthreads();
    if (!*s_flag) return;
    __threadfence();
    constexpr int CS = 2 * kG8MaxSplits + 2 + kG8MaxSplits + 1;   // floats per head
    float* scratch = reinterpret_cast<float*>(smem + L.tile);
    if (warp < G) {
        float* cw = scratch + warp * CS;
        int* act = reinterpret_cast<int*>(cw + 2 * kG8MaxSplits + 2);
        const float* pb = p.part + ((size_t)b * p.Hq + h0 + warp) * splits * (2 * D + 4);
        combine_weights<D>(pb, active, cw, cw + 2 * kG8MaxSplits, lane, act, act + kG8MaxSplits);
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += NT) {
        const int h = i / D, d = i - h * D;
        const float* cw = scratch + h * CS;
        const float* cl = cw + 2 * kG8MaxSplits;
        const int* act = reinterpret_cast<const int*>(cw + 2 * kG8MaxSplits + 2);
        const int nact = act[kG8MaxSplits];
        const float* pb = p.part + ((size_t)b * p.Hq + h0 + h) * splits * (2 * D + 4);
        f2 acc = {0.0f, 0.0f};
        for (int k = 0; k < nact; ++k) {
            const int sp = act[k];
            const float* q = pb + (size_t)sp * (2 * D + 4);
            acc = f2_add(acc, f2_mul(f2{__ldcg(q + d), __ldcg(q + D + d)}, f2{cw[2 * sp], cw[2 * sp + 1]}));
        }
        const f2 l = {cl[0], cl[1]};
        p.out[((size_t)b * p.Hq + h0 + h) * D + d] =
            l.hi > 0.0f ? f2_to_bf16(f2_div(acc, l)) : __float2bfloat16_rn(0.0f);
    }
}

// Prefill pre-pass over the INT8 cache: one CTA per row, warp w handles KV
// heads w, w + 8, ...: the row's new K (per-head RMSNorm and RoPE, the
// attention's own code) and V quantised per head row into the row's slot.
constexpr int kPrepI8Threads = 256;
template <int D>
__global__ void __launch_bounds__(kPrepI8Threads) kv_prep_i8_kernel(const AttnI8Params P) {
    const AttnParams& p = P.a;
    constexpr int E = D / 32;
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int max_ctx = p.max_blocks * p.page;
    const int ctx_raw = p.ctx_lens[b];
    const bool bad_ctx = ctx_raw < 0 || ctx_raw > max_ctx;
    const int pos = ctx_raw - 1;
    const bool bad_pos = !bad_ctx && ctx_raw > 0 && pos >= p.max_pos;
    const bool live = !bad_ctx && !bad_pos && ctx_raw > 0;
    HeadPre<D> hp;
    if (live) load_head_pre<D>(p, pos, lane, hp);
    pdl_wait();
    pdl_trigger();
    if (!live) return;   // the attention kernel flags bad contexts and positions
    const long slot = p.slot_mapping[b];
    const long num_slots = (long)p.num_blocks * p.page;
    if (threadIdx.x == 0 && slot >= num_slots) set_error(p.err, 0x1u);
    const bool slot_ok = slot >= 0 && slot < num_slots;
    const int NQ = p.Hq * D, NK = p.Hkv * D;
    const bf16* row = p.q + (size_t)b * p.q_stride;
    for (int kvh = warp; kvh < p.Hkv; kvh += kPrepI8Threads / 32) {
        float x[E], vv[E], y[E];
        load_bf16_lane<D>(row + NQ + (size_t)kvh * D + lane * E, x);
        load_bf16_lane<D>(row + NQ + NK + (size_t)kvh * D + lane * E, vv);
        norm_rope_head<D>(x, hp.kw, hp, p.eps, lane, y);
        int kc[E], vc[E];
        const float ks = quant_row_warp<E>(y, kc);
        const float vs = quant_row_warp<E>(vv, vc);
        if (slot_ok && lane == 0) {
            P.k_scale[(size_t)slot * p.Hkv + kvh] = ks;
            P.v_scale[(size_t)slot * p.Hkv + kvh] = vs;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            if (slot_ok) {
                P.k_codes[((size_t)slot * p.Hkv + kvh) * D + d] = (int8_t)kc[e];
                P.v_codes[((size_t)slot * p.Hkv + kvh) * D + d] = (int8_t)vc[e];
            }
            if (p.tap_k_rot) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = f2bf(y[e]);
        }
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_i8(Kern kern, dim3 grid, dim3 block, size_t smem, const Launch& L,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D>
cudaError_t launch_attn_i8_d(const AttnI8Params& P, const Launch& L) {
    const AttnParams& p = P.a;
    const int max_ctx = p.max_blocks * p.page;
    const bool in_kernel = in_kernel_combine(max_ctx, p.tickets != nullptr);
    const int chunk = attn_chunk(max_ctx, in_kernel);
    const int splits = attn_splits(max_ctx, in_kernel);
    const size_t smem = i8_item_smem_bytes(chunk, D);
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(attn_i8_kernel<D>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(attn_i8_kernel<D>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)i8_item_smem_bytes(256, 128));
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    if (smem > i8_item_smem_bytes(256, 128)) return cudaErrorInvalidValue;
    AttnI8Params q = P;
    if (!in_kernel) q.a.tickets = nullptr;
    cudaError_t e = launch_i8(attn_i8_kernel<D>, dim3(splits, p.Hq, p.B), dim3(kAttnThreads), smem,
                              L, q, chunk, splits);
    if (e != cudaSuccess || splits == 1 || in_kernel) return e;
    if ((size_t)(2 * splits + 2) * sizeof(float) > 48 * 1024) return cudaErrorInvalidValue;
    return launch_i8(attn_i8_combine_kernel<D>, dim3(p.Hq, p.B), dim3(D),
                     (size_t)(2 * splits + 2) * sizeof(float), L, (const float*)p.part, splits, p.Hq,
                     p.out);
}

template <int D, int G>
cudaError_t launch_g8_t(const AttnI8Params& P, int splits, const Launch& L) {
    const size_t smem = g8_smem(D, G).total;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(attn_i8_group_kernel<D, G>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(attn_i8_group_kernel<D, G>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    return launch_i8(attn_i8_group_kernel<D, G>, dim3(splits, P.a.Hkv, P.a.B), dim3(kG8Threads),
                     smem, L, P, splits);
}

template <int D>
cudaError_t launch_g8_d(const AttnI8Params& P, int splits, const Launch& L) {
    switch (P.a.Hq / P.a.Hkv) {
        case 1: return launch_g8_t<D, 1>(P, splits, L);
        case 2: return launch_g8_t<D, 2>(P, splits, L);
        case 3: return launch_g8_t<D, 3>(P, splits, L);
        case 4: return launch_g8_t<D, 4>(P, splits, L);
        case 5: return launch_g8_t<D, 5>(P, splits, L);
        case 6: return launch_g8_t<D, 6>(P, splits, L);
        case 7: return launch_g8_t<D, 7>(P, splits, L);
        default: return cudaErrorInvalidValue;
    }
}

// Decode-layer attention over at least this many (request, cached token)
// slots of the launch shape uses the grouped form (as for the BF16 cache).
constexpr long kG8MinWork = 8192;

}  // namespace

cudaError_t launch_attention_i8(const AttnI8Params& P, const Launch& L) {
    const AttnParams& p = P.a;
    if (p.B == 0) return cudaSuccess;
    const int max_ctx = p.max_blocks * p.page;
    const bool grouped_ok = p.fused && p.tickets && attn_group_shape_ok(p.Hq, p.Hkv, p.D, max_ctx);
    if (p.kv_in_cache && !grouped_ok) return cudaErrorInvalidValue;   // prefill: grouped form only
    if (grouped_ok && (p.kv_in_cache || (long)p.B * max_ctx >= kG8MinWork)) {
        const int splits = (max_ctx + kG8Chunk - 1) / kG8Chunk;
        if (splits > kG8MaxSplits) return cudaErrorInvalidValue;
        return p.D == 128 ? launch_g8_d<128>(P, splits, L) : launch_g8_d<64>(P, splits, L);
    }
    if (p.D == 128) return launch_attn_i8_d<128>(P, L);
    if (p.D == 64) return launch_attn_i8_d<64>(P, L);
    return cudaErrorInvalidValue;
}

cudaError_t launch_kv_prep_i8(const AttnI8Params& P, const Launch& L) {
    if (P.a.B == 0) return cudaSuccess;
    if (!P.a.fused || (P.a.D != 128 && P.a.D != 64)) return cudaErrorInvalidValue;
    if (P.a.D == 128)
        return launch_i8(kv_prep_i8_kernel<128>, dim3(P.a.B), dim3(kPrepI8Threads), 0, L, P);
    return launch_i8(kv_prep_i8_kernel<64>, dim3(P.a.B), dim3(kPrepI8Threads), 0, L, P);
}

cudaError_t launch_kv_write_i8(const bf16* k, const bf16* v, int T, int Hkv, int D,
                               const int32_t* slot_mapping, int8_t* k_codes, int8_t* v_codes,
                               float* k_scale, float* v_scale, long num_slots, unsigned* err,
                               const Launch& L) {
    if (T == 0) return cudaSuccess;
    const long rows = (long)T * Hkv;
    const int blocks = (int)((rows + 7) / 8);
    if (D == 128)
        return launch_i8(kv_write_i8_kernel<128>, dim3(blocks), dim3(256), 0, L, k, v, T, Hkv,
                         slot_mapping, k_codes, v_codes, k_scale, v_scale, num_slots, err);
    if (D == 64)
        return launch_i8(kv_write_i8_kernel<64>, dim3(blocks), dim3(256), 0, L, k, v, T, Hkv,
                         slot_mapping, k_codes, v_codes, k_scale, v_scale, num_slots, err);
    return cudaErrorInvalidValue;
}

}  // namespace a8w8
