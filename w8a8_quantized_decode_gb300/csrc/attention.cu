// attention.cu -- paged BF16 KV write and GQA decode attention (split-KV).
//
// "perf(qwen3-a8w8): optimize decode scheduling and data paths" (pypto-lib PR
// #810), "BF16 KV cache": K/V are stored in BF16 with no scale tensors and
// attention loads them directly; "Add Qwen3 A8W8 L2 runner foundation"
// (pypto-serving PR #61), "Summary": block table and slot mapping address the
// pages. "[Feature] Add native Qwen3-14B A8W8 serving path" (pypto-serving
// issue #52), "Current behavior": the decode layer normalises Q and K per head
// and applies RoPE before attention ("fused QK norm path").
//
// One CTA handles one (request, KV head, token chunk). It serves the whole GQA
// group of Hq/Hkv query heads, so every cached K/V byte is read once.
//   1. Before griddepcontrol.wait: the chunk's cached K and V rows (earlier
//      tokens, immutable during this kernel's predecessors) are copied into
//      shared memory with cp.async, so the KV read overlaps the tail of the
//      QKV projection.
//   2. Fused prologue (decode layer): per-head RMSNorm of the G query heads
//      and of the new K head (float32, rounded to BF16), rotate-half RoPE at
//      position ctx_len - 1 from a cos/sin table (rounded to BF16); the CTA
//      whose chunk holds the new token writes K/V into the cache slot and
//      into its shared tiles.
//   3. Scores: D/8 lanes per token, 8 BF16 of K per lane, the G query heads
//      in registers, reduced over the lane group with shuffles.
//   4. Softmax per head over the chunk (max-subtracted, float32).
//   5. P.V with column pairs per thread, reduced over token groups.
//   6. One chunk: normalise and write BF16. Several chunks: write float32
//      partials (unnormalised o, running max m, sum l) and combine them in a
//      second kernel: O = sum_s o_s e^{m_s - M} / sum_s l_s e^{m_s - M}.
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kGMax = 8;

size_t attn_smem_bytes(int chunk, int D) {
    return (size_t)2 * chunk * D * 2 + (size_t)kGMax * D * 4 + (size_t)kGMax * chunk * 4 +
           (size_t)kGMax * 2 * 4;
}

// Per-head RMSNorm + RoPE of one head vector held as E = D/32 elements per
// lane (elements [lane*E, lane*E + E)); the rotate-half partner of lane l is
// lane l ^ 16. Returns BF16-rounded results in y.
template <int D>
__device__ __forceinline__ void norm_rope_head(const bf16* src, const bf16* norm_w,
                                               const float* rope_row, float eps, int lane,
                                               float (&y)[D / 32]) {
    constexpr int E = D / 32;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = bf2f(src[lane * E + e]);
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss += x[e] * x[e];
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), eps)));
#pragma unroll
    for (int e = 0; e < E; ++e)
        x[e] = bf2f(f2bf(__fmul_rn(__fmul_rn(x[e], inv), bf2f(norm_w[lane * E + e]))));
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
        const int i = (lane * E + e) % (D / 2);
        const float c = rope_row[i], s = rope_row[D / 2 + i];
        float r;
        if (lane < 16) r = __fsub_rn(__fmul_rn(x[e], c), __fmul_rn(partner, s));
        else r = __fadd_rn(__fmul_rn(x[e], c), __fmul_rn(partner, s));
        y[e] = bf2f(f2bf(r));
    }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnParams p, int chunk,
                                                            int splits) {
    extern __shared__ __align__(16) unsigned char smem[];
    bf16* Ks = reinterpret_cast<bf16*>(smem);
    bf16* Vs = Ks + (size_t)chunk * D;
    float* qs = reinterpret_cast<float*>(Vs + (size_t)chunk * D);
    float* sc = qs + kGMax * D;
    float* stat = sc + (size_t)kGMax * chunk;
    float* red = reinterpret_cast<float*>(smem);   // aliases Ks once the scores are done
    __shared__ int s_bad_block;

    const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.Hq / p.Hkv;
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

    if (threadIdx.x == 0) s_bad_block = 0;
    __syncthreads();
    constexpr int RV = D / 8;   // 16-byte vectors per row
    for (int i = threadIdx.x; i < n_old * RV; i += kAttnThreads) {
        const int t = i / RV, c = i - t * RV;
        const int tok = t0 + t;
        const int blk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        if (blk < 0 || blk >= p.num_blocks) {
            *reinterpret_cast<int4*>(Ks + (size_t)t * D + 8 * c) = make_int4(0, 0, 0, 0);
            *reinterpret_cast<int4*>(Vs + (size_t)t * D + 8 * c) = make_int4(0, 0, 0, 0);
            s_bad_block = 1;
            continue;
        }
        const size_t off = (((size_t)blk * p.page + tok % p.page) * p.Hkv + kvh) * D + 8 * c;
        cp_async16(Ks + (size_t)t * D + 8 * c, p.k_cache + off);
        cp_async16(Vs + (size_t)t * D + 8 * c, p.v_cache + off);
    }
    cp_async_commit();

    pdl_wait();
    pdl_trigger();

    if (threadIdx.x == 0) {
        if (bad_ctx) set_error(p.err, 0x4u);
        if (bad_pos) set_error(p.err, 0x10u);
    }

    // query heads (and, for the CTA holding the new token, its K and V)
    if (n > 0) {
        for (int task = warp; task <= G; task += kAttnWarps) {
            if (task < G) {
                const int h = kvh * G + task;
                const bf16* src = p.q + (size_t)b * p.q_stride + (size_t)h * D;
                constexpr int E = D / 32;
                float y[E];
                if (p.fused) {
                    norm_rope_head<D>(src, p.q_norm_w, p.rope + (size_t)pos * D, p.eps, lane, y);
                    if (p.tap_q_rot && split == 0) {
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            p.tap_q_rot[((size_t)b * p.Hq + h) * D + lane * E + e] = f2bf(y[e]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) y[e] = bf2f(src[lane * E + e]);
                }
#pragma unroll
                for (int e = 0; e < E; ++e) qs[task * D + lane * E + e] = y[e];
            } else if (covers_new) {
                constexpr int E = D / 32;
                const int NQ = p.Hq * D, NK = p.Hkv * D;
                const bf16* ksrc = p.q + (size_t)b * p.q_stride + NQ + (size_t)kvh * D;
                const bf16* vsrc = p.q + (size_t)b * p.q_stride + NQ + NK + (size_t)kvh * D;
                float y[E];
                norm_rope_head<D>(ksrc, p.k_norm_w, p.rope + (size_t)pos * D, p.eps, lane, y);
                const int tr = pos - t0;
                const long slot = p.slot_mapping[b];
                const long num_slots = (long)p.num_blocks * p.page;
                const bool slot_ok = slot >= 0 && slot < num_slots;
                if (lane == 0 && slot >= num_slots) set_error(p.err, 0x1u);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int d = lane * E + e;
                    const bf16 kb = f2bf(y[e]);
                    const bf16 vb = vsrc[d];
                    Ks[(size_t)tr * D + d] = kb;
                    Vs[(size_t)tr * D + d] = vb;
                    if (slot_ok) {
                        p.k_cache[((size_t)slot * p.Hkv + kvh) * D + d] = kb;
                        p.v_cache[((size_t)slot * p.Hkv + kvh) * D + d] = vb;
                    }
                    if (p.tap_k_rot) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = kb;
                }
            }
        }
    }
    cp_async_wait_all();
    __syncthreads();
    if (threadIdx.x == 0 && s_bad_block) set_error(p.err, 0x2u);

    // scores
    constexpr int LPT = D / 8;
    constexpr int TPW = 32 / LPT;
    const int j = lane % LPT, tw = lane / LPT;
    if (n > 0) {
        float qr[kGMax][8];
#pragma unroll
        for (int g = 0; g < kGMax; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) qr[g][e] = (g < G) ? qs[g * D + 8 * j + e] : 0.0f;
        const int step = kAttnWarps * TPW;
        const int n_pad = ((n + step - 1) / step) * step;
        for (int t = warp * TPW + tw; t < n_pad; t += step) {
            float kf[8];
            if (t < n) {
                unpack8(*reinterpret_cast<const int4*>(Ks + (size_t)t * D + 8 * j), kf);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) kf[e] = 0.0f;
            }
#pragma unroll
            for (int g = 0; g < kGMax; ++g) {
                if (g < G) {
                    float d = 0.0f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) d = fmaf(qr[g][e], kf[e], d);
#pragma unroll
                    for (int o = LPT / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                    if (j == 0 && t < n) sc[g * chunk + t] = d * p.scale;
                }
            }
        }
    }
    __syncthreads();

    // softmax over the chunk, per head
    for (int g = warp; g < G; g += kAttnWarps) {
        float m = -INFINITY;
        for (int t = lane; t < n; t += 32) m = fmaxf(m, sc[g * chunk + t]);
        m = warp_max(m);
        float l = 0.0f;
        for (int t = lane; t < n; t += 32) {
            const float e = expf(sc[g * chunk + t] - m);
            sc[g * chunk + t] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            stat[2 * g] = m;
            stat[2 * g + 1] = l;
        }
    }
    __syncthreads();

    // P.V: thread = (column pair, token group)
    constexpr int CP = D / 2;
    constexpr int NTG = kAttnThreads / CP;
    const int cp = threadIdx.x % CP, tg = threadIdx.x / CP;
    float o[kGMax][2];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) o[g][0] = o[g][1] = 0.0f;
    for (int t = tg; t < n; t += NTG) {
        const float2 v = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(Vs + (size_t)t * D + 2 * cp));
#pragma unroll
        for (int g = 0; g < kGMax; ++g) {
            if (g < G) {
                const float pr = sc[g * chunk + t];
                o[g][0] = fmaf(pr, v.x, o[g][0]);
                o[g][1] = fmaf(pr, v.y, o[g][1]);
            }
        }
    }
    // Ks is no longer read: reuse it for the cross-group reduction
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
        if (g < G) {
            red[((size_t)tg * kGMax + g) * D + 2 * cp] = o[g][0];
            red[((size_t)tg * kGMax + g) * D + 2 * cp + 1] = o[g][1];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += kAttnThreads) {
        const int g = i / D, d = i - g * D;
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < NTG; ++q) acc += red[((size_t)q * kGMax + g) * D + d];
        const int h = kvh * G + g;
        if (splits == 1) {
            const float val = n > 0 ? __fdiv_rn(acc, stat[2 * g + 1]) : 0.0f;
            p.out[((size_t)b * p.Hq + h) * D + d] = f2bf(val);
        } else {
            float* pp = p.part + (((size_t)b * p.Hq + h) * splits + split) * (D + 2);
            pp[d] = n > 0 ? acc : 0.0f;
            if (d == 0) {
                pp[D] = n > 0 ? stat[2 * g] : -INFINITY;
                pp[D + 1] = n > 0 ? stat[2 * g + 1] : 0.0f;
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const float* __restrict__ part, int splits,
                                                         int Hq, bf16* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const float* pp = part + ((size_t)b * Hq + h) * splits * (D + 2);
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, pp[(size_t)s * (D + 2) + D]);
    float L = 0.0f, acc = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float m = pp[(size_t)s * (D + 2) + D];
            if (m == -INFINITY) continue;
            const float w = expf(m - M);
            L = fmaf(pp[(size_t)s * (D + 2) + D + 1], w, L);
            acc = fmaf(pp[(size_t)s * (D + 2) + d], w, acc);
        }
    }
    out[((size_t)b * Hq + h) * D + d] = f2bf(L > 0.0f ? __fdiv_rn(acc, L) : 0.0f);
}

__global__ void kv_write_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v, int T,
                                int row_vec, const int32_t* __restrict__ slot_mapping,
                                bf16* __restrict__ k_cache, bf16* __restrict__ v_cache,
                                long num_slots, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)T * row_vec) return;
    const int t = (int)(i / row_vec), c = (int)(i - (long)t * row_vec);
    const long slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (c == 0) set_error(err, 0x1u);
        return;
    }
    const int4 kv = ld_nc_v4(k + ((size_t)t * row_vec + c) * 8);
    const int4 vv = ld_nc_v4(v + ((size_t)t * row_vec + c) * 8);
    *reinterpret_cast<int4*>(k_cache + ((size_t)slot * row_vec + c) * 8) = kv;
    *reinterpret_cast<int4*>(v_cache + ((size_t)slot * row_vec + c) * 8) = vv;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, const Launch& L,
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
cudaError_t launch_attn_d(const AttnParams& p, const Launch& L) {
    const int max_ctx = p.max_blocks * p.page;
    const int chunk = attn_chunk(max_ctx);
    const int splits = attn_splits(max_ctx);
    const size_t smem = attn_smem_bytes(chunk, D);
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)attn_smem_bytes(256, 128));
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    cudaError_t e = launch_ex(attn_kernel<D>, dim3(splits, p.Hkv, p.B), dim3(kAttnThreads), smem,
                              L, p, chunk, splits);
    if (e != cudaSuccess || splits == 1) return e;
    return launch_ex(attn_combine_kernel<D>, dim3(p.Hq, p.B), dim3(D), 0, L,
                     (const float*)p.part, splits, p.Hq, p.out);
}

}  // namespace

int attn_chunk(int max_ctx) { return max_ctx <= 256 ? 256 : 128; }

int attn_splits(int max_ctx) {
    const int c = attn_chunk(max_ctx);
    return max_ctx <= 0 ? 1 : (max_ctx + c - 1) / c;
}

size_t attn_part_bytes(int B, int Hq, int D, int max_ctx) {
    const int s = attn_splits(max_ctx);
    if (s <= 1) return 0;
    return (size_t)B * Hq * s * (D + 2) * sizeof(float);
}

cudaError_t launch_attention(const AttnParams& p, const Launch& L) {
    if (p.B == 0) return cudaSuccess;
    if (p.D == 128) return launch_attn_d<128>(p, L);
    if (p.D == 64) return launch_attn_d<64>(p, L);
    return cudaErrorInvalidValue;
}

cudaError_t launch_kv_write(const bf16* k, const bf16* v, int T, int Hkv, int D,
                            const int32_t* slot_mapping, bf16* k_cache, bf16* v_cache,
                            long num_slots, unsigned* err, const Launch& L) {
    if (T == 0) return cudaSuccess;
    const int row_vec = Hkv * D / 8;
    const long total = (long)T * row_vec;
    const int threads = 256;
    const int blocks = (int)((total + threads - 1) / threads);
    return launch_ex(kv_write_kernel, dim3(blocks), dim3(threads), 0, L, k, v, T, row_vec,
                     slot_mapping, k_cache, v_cache, num_slots, err);
}

}  // namespace a8w8
