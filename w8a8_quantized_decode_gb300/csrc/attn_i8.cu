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
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(attn_i8_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)i8_item_smem_bytes(256, 128));
        if (e != cudaSuccess) return e;
        configured_dev = dev;
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

}  // namespace

cudaError_t launch_attention_i8(const AttnI8Params& P, const Launch& L) {
    if (P.a.B == 0) return cudaSuccess;
    if (P.a.D == 128) return launch_attn_i8_d<128>(P, L);
    if (P.a.D == 64) return launch_attn_i8_d<64>(P, L);
    return cudaErrorInvalidValue;
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
