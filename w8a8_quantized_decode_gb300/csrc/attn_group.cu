// attn_group.cu -- paged GQA decode attention for large batches and long
// contexts: one CTA per (request, KV head, 128-token chunk) serving every
// query head of the group.
//
// Same method and arithmetic as attn_impl.cuh ("perf(qwen3-a8w8): optimize
// decode scheduling and data paths", pypto-lib PR #810, "BF16 KV cache";
// "[Feature] Add native Qwen3-14B A8W8 serving path", pypto-serving issue #52,
// "Current behavior": per-head QK RMSNorm and RoPE before attention): scores
// q.k / sqrt(D) of BF16 operands, max-subtracted softmax, P.V, all evaluated
// in two-float arithmetic so that the BF16 output is the correctly rounded
// value of the real-valued result.
//
// Why a second form: with two-float arithmetic attention is ALU bound. The
// per-query-head form (attn_impl.cuh) suits batch-1 decode (many small CTAs,
// short latency); at batch 16 and contexts of thousands of tokens it spends
// most of its instructions on shuffle reductions, a one-warp softmax and
// staging every K/V tile once per query head. Here:
//   * the K tile of the chunk is staged once for the G = Hq / Hkv query
//     heads of the KV head (cp.async, before the dependency wait), and the V
//     tile replaces it in the same buffer while the softmax runs, so that
//     five CTAs fit on an SM;
//   * scores: one lane per token, the lane's K row read from shared memory
//     8 columns at a time and multiplied with the query rows (broadcast
//     reads) of the warp's heads; products of BF16 values are exact in
//     float32 and summed as (hi, lo) pairs (TwoSum), with no reduction;
//   * softmax: one warp per head;
//   * P.V: thread (column pair, token group) accumulates all heads of the
//     group, each term p * v as an exact product pair added by TwoSum with
//     the low parts summed separately (Ogita, Rump and Oishi's Dot2), then
//     the token groups are combined with shuffles;
//   * more than one chunk: two-float partials (o, m, l) per head, merged by
//     the last CTA of the (request, KV head) to finish (atomic ticket).
#include "attn_impl.cuh"

namespace a8w8 {

namespace {

constexpr int kGrpThreads = 256;
constexpr int kGrpChunk = 128;
constexpr int kGrpMaxG = 7;          // query heads per KV head served here
constexpr int kGrpMaxSplits = 64;    // chunks per request (in-kernel combine)

struct GrpSmem {
    size_t tile, vnew, q, pr, stat, blk, flag, total;
};
__host__ __device__ inline GrpSmem grp_smem(int D, int G) {
    GrpSmem s;
    s.tile = 0;
    const size_t kv = (size_t)kGrpChunk * (D + kTilePad) * 2;
    // combine scratch reuses the tile: per head 2*splits weights, 2 for L,
    // splits active indices and their count
    const size_t comb = (size_t)G * (2 * kGrpMaxSplits + 2 + kGrpMaxSplits + 1) * 4;
    s.vnew = (kv > comb ? kv : comb);                    // [D] bf16: the new token's V
    s.q = s.vnew + (size_t)D * 2;                        // [G][D] float
    s.pr = s.q + (size_t)G * D * 4;                      // [G][chunk] (hi, lo) pairs
    s.stat = s.pr + (size_t)G * kGrpChunk * 8;           // [G][4]: m hi, m lo, l hi, l lo
    s.blk = s.stat + (size_t)G * 4 * 4;                  // [chunk] physical block per token
    s.flag = s.blk + (size_t)kGrpChunk * 4;
    s.total = s.flag + 16;
    return s;
}

// acc += p * v with p a pair and v a float: the product's high part is added
// by TwoSum, its rounding error, p.lo * v and the TwoSum error go to acc.lo
// (no renormalisation per term).
__device__ __forceinline__ void dot2_acc(f2& acc, const f2 p, float v) {
    const float h = __fmul_rn(p.hi, v);
    const float e = __fmaf_rn(p.hi, v, -h);
    float s, err;
    two_sum(acc.hi, h, s, err);
    acc.hi = s;
    acc.lo = __fadd_rn(acc.lo, __fadd_rn(err, __fmaf_rn(p.lo, v, e)));
}

template <int D, int G>
__global__ void __launch_bounds__(kGrpThreads) attn_group_kernel(const AttnParams p, int splits) {
    static_assert(G >= 1 && G <= kGrpMaxG, "query heads per KV head");
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NT = kGrpThreads, C = kGrpChunk;
    constexpr int DP = D + kTilePad;
    constexpr int RV = D / 8;         // 16-byte vectors per row
    constexpr int E = D / 32;
    const GrpSmem L = grp_smem(D, G);
    bf16* Ts = reinterpret_cast<bf16*>(smem + L.tile);   // K tile, then V tile
    bf16* vnew = reinterpret_cast<bf16*>(smem + L.vnew);
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

    // physical block of every cached token of the chunk
    if (tid == 0) *s_flag = 0;
    for (int t = tid; t < n_old; t += NT) {
        const int tok = t0 + t;
        const int bk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        blk[t] = (bk < 0 || bk >= p.num_blocks) ? -1 : bk;
    }
    // prefill: the cache rows of this launch's tokens are written by the
    // kernel before, so they are read only after the dependency wait
    if (p.kv_in_cache) pdl_wait();
    __syncthreads();
    // rows of the cached tokens of `cache` into the tile (zeros for a bad block)
    auto load_tile = [&](const bf16* cache) {
        for (int i = tid; i < n_old * RV; i += NT) {
            const int t = i / RV, c = i - t * RV;
            const int bk = blk[t];
            if (bk < 0) {
                *reinterpret_cast<int4*>(Ts + (size_t)t * DP + 8 * c) = make_int4(0, 0, 0, 0);
                *s_flag = 1;
                continue;
            }
            const int tok = t0 + t;
            const size_t off = (((size_t)bk * p.page + tok % p.page) * p.Hkv + kvh) * D + 8 * c;
            cp_async16(Ts + (size_t)t * DP + 8 * c, cache + off);
        }
        cp_async_commit();
    };
    load_tile(p.k_cache);
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
        const int tr = pos - t0;
        const long slot = p.slot_mapping[b];
        const long num_slots = (long)p.num_blocks * p.page;
        const bool slot_ok = slot >= 0 && slot < num_slots;
        if (lane == 0 && slot >= num_slots && !p.kv_in_cache) set_error(p.err, 0x1u);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            const bf16 kb = f2bf(y[e]);
            const bf16 vb = f2bf(vv[e]);
            Ts[(size_t)tr * DP + d] = kb;
            vnew[d] = vb;
            if (slot_ok && !p.kv_in_cache) {
                p.k_cache[((size_t)slot * p.Hkv + kvh) * D + d] = kb;
                p.v_cache[((size_t)slot * p.Hkv + kvh) * D + d] = vb;
            }
            if (p.tap_k_rot && !p.kv_in_cache) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = kb;
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
            const bf16* krow = Ts + (size_t)t * DP;
#pragma unroll 2
            for (int dv = 0; dv < RV; ++dv) {
                float kf[8];
                unpack8(*reinterpret_cast<const int4*>(krow + 8 * dv), kf);
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
                    const f2 sv = f2_mul(fast_two_sum(acc[i].hi, acc[i].lo), scale);
                    pr[hh * C + t] = make_float2(sv.hi, sv.lo);
                }
            }
        }
    }
    __syncthreads();   // the K tile is no longer read

    // the V tile into the same buffer, behind the softmax
    load_tile(p.v_cache);
    if (n > 0 && warp == G && covers_new) {
        for (int d = lane; d < D; d += 32) Ts[(size_t)(pos - t0) * DP + d] = vnew[d];
    }

    // softmax of head w over the chunk: p = exp(s - m), l = sum p
    if (warp < G) {
        float2* ph = pr + warp * C;
        f2 m = {-INFINITY, 0.0f};
        for (int t = lane; t < n; t += 32) m = f2_max(m, f2{ph[t].x, ph[t].y});
        m = warp_max_f2(m);
        f2 l = {0.0f, 0.0f};
        for (int t = lane; t < n; t += 32) {
            const f2 e = f2_exp(f2_sub(f2{ph[t].x, ph[t].y}, m));
            ph[t] = make_float2(e.hi, e.lo);
            l = f2_add(l, e);
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
            const float2 v = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162*>(Ts + (size_t)t * DP + 2 * cp));
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 q = pr[h * C + t];
                dot2_acc(o[h][0], f2{q.x, q.y}, v.x);
                dot2_acc(o[h][1], f2{q.x, q.y}, v.y);
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            {
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
        }
        if (tg == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                {
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
    constexpr int CS = 2 * kGrpMaxSplits + 2 + kGrpMaxSplits + 1;   // floats per head
    float* scratch = reinterpret_cast<float*>(smem + L.tile);
    if (warp < G) {
        float* cw = scratch + warp * CS;
        int* act = reinterpret_cast<int*>(cw + 2 * kGrpMaxSplits + 2);
        const float* pb = p.part + ((size_t)b * p.Hq + h0 + warp) * splits * (2 * D + 4);
        combine_weights<D>(pb, active, cw, cw + 2 * kGrpMaxSplits, lane, act, act + kGrpMaxSplits);
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += NT) {
        const int h = i / D, d = i - h * D;
        const float* cw = scratch + h * CS;
        const float* cl = cw + 2 * kGrpMaxSplits;
        const int* act = reinterpret_cast<const int*>(cw + 2 * kGrpMaxSplits + 2);
        const int nact = act[kGrpMaxSplits];
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

// Prefill pre-pass: one CTA per row, warp w handles KV heads w, w + 8, ...:
// per-head RMSNorm and RoPE of the row's new K (the attention's own code),
// then K and V into the row's cache slot.
constexpr int kPrepKvThreads = 256;
template <int D>
__global__ void __launch_bounds__(kPrepKvThreads) kv_prep_kernel(const AttnParams p) {
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
    for (int kvh = warp; kvh < p.Hkv; kvh += kPrepKvThreads / 32) {
        float x[E], vv[E], y[E];
        load_bf16_lane<D>(row + NQ + (size_t)kvh * D + lane * E, x);
        load_bf16_lane<D>(row + NQ + NK + (size_t)kvh * D + lane * E, vv);
        norm_rope_head<D>(x, hp.kw, hp, p.eps, lane, y);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            const bf16 kb = f2bf(y[e]);
            if (slot_ok) {
                p.k_cache[((size_t)slot * p.Hkv + kvh) * D + d] = kb;
                p.v_cache[((size_t)slot * p.Hkv + kvh) * D + d] = f2bf(vv[e]);
            }
            if (p.tap_k_rot) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = kb;
        }
    }
}

}  // namespace

cudaError_t launch_kv_prep(const AttnParams& p, const Launch& L) {
    if (p.B == 0) return cudaSuccess;
    if (!p.fused || (p.D != 128 && p.D != 64)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B);
    cfg.blockDim = dim3(kPrepKvThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    if (p.D == 128) return cudaLaunchKernelEx(&cfg, kv_prep_kernel<128>, p);
    return cudaLaunchKernelEx(&cfg, kv_prep_kernel<64>, p);
}

bool attn_group_shape_ok(int Hq, int Hkv, int D, int max_ctx) {
    return Hkv > 0 && Hq % Hkv == 0 && Hq / Hkv <= kGrpMaxG && (D == 128 || D == 64) &&
           (max_ctx + kGrpChunk - 1) / kGrpChunk <= kGrpMaxSplits;
}

bool attn_group_supported(const AttnParams& p) {
    return p.fused && p.tickets && attn_group_shape_ok(p.Hq, p.Hkv, p.D, p.max_blocks * p.page);
}

int attn_group_splits(int max_ctx) { return max_ctx <= 0 ? 1 : (max_ctx + kGrpChunk - 1) / kGrpChunk; }

template <int D, int G>
cudaError_t launch_grp_t(const AttnParams& p, int splits, const Launch& L) {
    const size_t smem = grp_smem(D, G).total;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(attn_group_kernel<D, G>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(attn_group_kernel<D, G>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits, p.Hkv, p.B);
    cfg.blockDim = dim3(kGrpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_group_kernel<D, G>, p, splits);
}

template <int D>
cudaError_t launch_grp_d(const AttnParams& p, int splits, const Launch& L) {
    switch (p.Hq / p.Hkv) {
        case 1: return launch_grp_t<D, 1>(p, splits, L);
        case 2: return launch_grp_t<D, 2>(p, splits, L);
        case 3: return launch_grp_t<D, 3>(p, splits, L);
        case 4: return launch_grp_t<D, 4>(p, splits, L);
        case 5: return launch_grp_t<D, 5>(p, splits, L);
        case 6: return launch_grp_t<D, 6>(p, splits, L);
        case 7: return launch_grp_t<D, 7>(p, splits, L);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_attn_group(const AttnParams& p, const Launch& L) {
    if (p.B == 0) return cudaSuccess;
    if (!attn_group_supported(p)) return cudaErrorInvalidValue;
    const int splits = attn_group_splits(p.max_blocks * p.page);
    if (p.D == 128) return launch_grp_d<128>(p, splits, L);
    return launch_grp_d<64>(p, splits, L);
}

}  // namespace a8w8
