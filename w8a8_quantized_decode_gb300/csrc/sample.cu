// sample.cu -- device-side sampling beyond greedy: temperature and top-p
// (nucleus) over a logits row, by the Gumbel-max rule.
//
// Reading of the serving step ("Add native Qwen3 14B A8W8 serving path",
// pypto-serving PR #48, "Performance": greedy decoding, temperature 0 and
// top_p 1; "Add Qwen3 A8W8 L2 runner foundation", pypto-serving PR #61,
// "Related": sampling on the device). Per row l:
//   T <= 0: argmax, lowest index on ties.
//   z = (l - max l) / T, p = exp(z); with p32 = float(p), the nucleus is
//   {p32 >= tau} for the largest tau among the p32 values whose tokens carry
//   at least top_p of the total mass (all of them for top_p >= 1); the token is
//   the argmax over the nucleus of z_i + g_i, g_i = -log(-log(u_i)), which is
//   a draw from softmax(z) restricted to the nucleus (Gumbel-max rule).
//   u_i = (floor(x / 2^8) + 1/2) / 2^24, x the first word of Philox4x32-10
//   (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011)
//   with key (seed lo, seed hi) and counter (i, row, step lo, step hi).
//
// Each row is spread over kChunks CTAs. The argmax (greedy or Gumbel) is an
// atomic maximum on (order-preserving key bits, inverted index); the last CTA
// of the row (ticket) writes the token. top-p finds tau exactly by a radix
// selection over the float bits of p32 (p in (0, 1]: bits <= 0x3f800000): the
// masses of three levels of 1024 buckets (bits 29..20, 19..10, 9..0) are
// summed as fixed-point integers (units of 2^-40, exact and order-free), each
// level's last CTA picks the bucket where the mass from the top reaches
// top_p * S; p and S are two-float values (S per CTA, summed in CTA order).
// The per-row state lives in the workspace and is cleared by the host before
// each call.
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kSampThreads = 256;
constexpr int kChunks = 64;                 // CTAs per row
constexpr int kBuckets = 1024;
constexpr double kFix = 1099511627776.0;    // 2^40

// Per-row state (cleared before each call); the workspace holds B states,
// then the rows' p values [B][V][2].
struct RowState {
    unsigned long long best;                 // packed argmax key
    unsigned maxbits;                        // order-preserving max logit
    unsigned tickets[5];
    unsigned sel[4];                         // level 1 / 2 buckets, tau bits
    float need_hi, need_lo;                  // top_p * S
    unsigned long long above;                // fixed-point mass above the current bucket
    float spart[2 * kChunks];                // per-CTA S (hi, lo)
    unsigned long long hist[3][kBuckets];
};
constexpr size_t kStateBytes = (sizeof(RowState) + 255) / 256 * 256;

__device__ __forceinline__ unsigned order_bits(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unorder_bits(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ unsigned long long pack_key(float v, int i) {
    return ((unsigned long long)order_bits(v) << 32) | (0xffffffffu - (unsigned)i);
}

__device__ __forceinline__ uint32_t mulhilo32(uint32_t a, uint32_t b, uint32_t& hi) {
    const unsigned long long p = (unsigned long long)a * b;
    hi = (uint32_t)(p >> 32);
    return (uint32_t)p;
}
// First output word of Philox4x32-10 for counter (c0, c1, c2, c3), key (k0, k1).
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint32_t hi0, hi1;
        const uint32_t lo0 = mulhilo32(0xD2511F53u, c0, hi0);
        const uint32_t lo1 = mulhilo32(0xCD9E8D57u, c2, hi1);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

struct SampArgs {
    const float* logits;
    int V, ld;
    float T, top_p;
    uint64_t seed, step;
    const uint64_t* step_ptr;   // when set, the step is read from here (captured graphs)
    unsigned char* ws;        // [B][kStateBytes], then [B][V][2] floats
    int32_t* out;
};

__device__ __forceinline__ RowState* row_state(const SampArgs& a, int b) {
    return reinterpret_cast<RowState*>(a.ws + (size_t)b * kStateBytes);
}
__device__ __forceinline__ float* row_p(const SampArgs& a, int b) {
    return reinterpret_cast<float*>(a.ws + (size_t)gridDim.y * kStateBytes + (size_t)b * a.V * 8);
}

// The last CTA of the row to arrive at ticket t returns true (after a fence).
__device__ __forceinline__ bool last_of_row(RowState* st, int t) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&st->tickets[t], 1u) == (unsigned)(kChunks - 1);
    __syncthreads();
    if (s_last) __threadfence();
    return s_last;
}

// Adds v into h[bucket] for the active lanes of a warp (every lane calls):
// lanes with the same bucket are summed first, so that each distinct bucket
// takes one shared-memory atomic per warp.
__device__ __forceinline__ void hist_add_warp(unsigned long long* h, unsigned bucket,
                                              unsigned long long v, bool active) {
    const unsigned key = active ? bucket : 0xffffffffu;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    unsigned long long sum = 0ull;
    for (unsigned m = peers; m; m &= m - 1) sum += __shfl_sync(peers, v, __ffs(m) - 1);
    if (active && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[bucket], sum);
}

// Run by the whole CTA: the bucket j of hist (descending order) where the
// mass from the top, starting at `above`, reaches nf; writes sel[level] and
// the mass above j. Thread t takes buckets 4t..4t+3; a suffix scan over the
// threads gives each its mass above.
__device__ __forceinline__ void pick_bucket(RowState* st, int level, unsigned long long nf) {
    __shared__ unsigned long long sums[kSampThreads];
    static_assert(kBuckets == 4 * kSampThreads, "4 buckets per thread");
    const int t = threadIdx.x;
    unsigned long long hb[4], own = 0ull;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        hb[k] = __ldcg(&st->hist[level][4 * t + k]);
        own += hb[k];
    }
    sums[t] = own;
    __syncthreads();
    // inclusive suffix sums: sums[t] = sum over t' >= t
    for (int d = 1; d < kSampThreads; d <<= 1) {
        const unsigned long long v = t + d < kSampThreads ? sums[t + d] : 0ull;
        __syncthreads();
        sums[t] += v;
        __syncthreads();
    }
    const unsigned long long base = __ldcg(&st->above);
    const unsigned long long hi_t = base + (t + 1 < kSampThreads ? sums[t + 1] : 0ull);  // above 4t+3
    // the crossing thread, or thread 0 when the total stays short of nf
    if (hi_t < nf && (hi_t + own >= nf || t == 0)) {
        unsigned long long cum = hi_t;
        int j = 4 * t + 3;
        for (; j > 4 * t; --j) {
            if (cum + hb[j - 4 * t] >= nf) break;
            cum += hb[j - 4 * t];
        }
        st->sel[level] = (unsigned)j;
        st->above = cum;
        if (level == 2) st->sel[3] = (st->sel[0] << 20) | (st->sel[1] << 10) | (unsigned)j;
    }
    // a row where the top bucket alone reaches nf: thread kSampThreads - 1
    // has hi_t = base < nf and crosses within its buckets (handled above)
}

// Block maximum of packed keys (each thread's candidate), then one atomicMax.
__device__ __forceinline__ void commit_best(RowState* st, unsigned long long k) {
    __shared__ unsigned long long red[kSampThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, k, o);
        k = x > k ? x : k;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = k;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long m = red[0];
        for (int w = 1; w < kSampThreads / 32; ++w) m = red[w] > m ? red[w] : m;
        atomicMax(&st->best, m);
    }
}

// Pass 1: row maximum (top-p only).
__global__ void __launch_bounds__(kSampThreads) samp_max_kernel(const SampArgs a) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y, c = blockIdx.x;
    const float* l = a.logits + (size_t)b * a.ld;
    const int i0 = (int)((long long)a.V * c / kChunks), i1 = (int)((long long)a.V * (c + 1) / kChunks);
    float m = -INFINITY;
    for (int i = i0 + threadIdx.x; i < i1; i += kSampThreads) m = fmaxf(m, __ldcg(l + i));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) atomicMax(&row_state(a, b)->maxbits, order_bits(m));
}

// Pass 2: p = exp((l - max) / T) (two-float) into the workspace, this CTA's S,
// level-1 histogram; the row's last CTA sums S and picks the level-1 bucket.
__global__ void __launch_bounds__(kSampThreads) samp_p_kernel(const SampArgs a) {
    __shared__ unsigned long long h[kBuckets];
    __shared__ float red[2 * (kSampThreads / 32)];
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y, c = blockIdx.x;
    RowState* st = row_state(a, b);
    float* pw = row_p(a, b);
    const float* l = a.logits + (size_t)b * a.ld;
    for (int j = threadIdx.x; j < kBuckets; j += kSampThreads) h[j] = 0ull;
    __syncthreads();
    const float mx = unorder_bits(__ldcg(&st->maxbits));
    const f2 tt = {a.T, 0.0f};
    const int i0 = (int)((long long)a.V * c / kChunks), i1 = (int)((long long)a.V * (c + 1) / kChunks);
    f2 S = {0.0f, 0.0f};
    for (int base = i0; base < i1; base += kSampThreads) {   // uniform trip count
        const int i = base + (int)threadIdx.x;
        const bool act = i < i1;
        f2 p = {0.0f, 0.0f};
        if (act) {
            float d, e;
            two_sum(__ldcg(l + i), -mx, d, e);   // l_i - max, exactly
            p = f2_exp(f2_div(f2{d, e}, tt));
            pw[2 * i] = p.hi;
            pw[2 * i + 1] = p.lo;
            S = f2_add(S, p);
        }
        const double pd = (double)p.hi + (double)p.lo;
        hist_add_warp(h, __float_as_uint(p.hi) >> 20, (unsigned long long)(pd * kFix), act);
    }
    S = warp_sum_f2(S);
    if ((threadIdx.x & 31) == 0) {
        red[2 * (threadIdx.x >> 5)] = S.hi;
        red[2 * (threadIdx.x >> 5) + 1] = S.lo;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        f2 t = {0.0f, 0.0f};
        for (int w = 0; w < kSampThreads / 32; ++w) t = f2_add(t, f2{red[2 * w], red[2 * w + 1]});
        st->spart[2 * c] = t.hi;
        st->spart[2 * c + 1] = t.lo;
    }
    for (int j = threadIdx.x; j < kBuckets; j += kSampThreads)
        if (h[j]) atomicAdd(&st->hist[0][j], h[j]);
    if (!last_of_row(st, 0)) return;
    __shared__ float sp[2 * kChunks];
    __shared__ unsigned long long s_nf;
    for (int k = threadIdx.x; k < 2 * kChunks; k += kSampThreads) sp[k] = __ldcg(&st->spart[k]);
    __syncthreads();
    if (threadIdx.x == 0) {
        f2 Stot = {0.0f, 0.0f};
        for (int k = 0; k < kChunks; ++k) Stot = f2_add(Stot, f2{sp[2 * k], sp[2 * k + 1]});
        const f2 need = f2_mulf(Stot, a.top_p);
        st->need_hi = need.hi;
        st->need_lo = need.lo;
        st->above = 0ull;
        s_nf = (unsigned long long)(((double)need.hi + (double)need.lo) * kFix);
    }
    __threadfence_block();
    __syncthreads();
    pick_bucket(st, 0, s_nf);
}

// Passes 3 and 4: histograms of the next 10 bits inside the chosen bucket;
// the last CTA picks the next bucket (level 3 fixes tau).
template <int LEVEL>
__global__ void __launch_bounds__(kSampThreads) samp_level_kernel(const SampArgs a) {
    __shared__ unsigned long long h[kBuckets];
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y, c = blockIdx.x;
    RowState* st = row_state(a, b);
    const float* pw = row_p(a, b);
    for (int j = threadIdx.x; j < kBuckets; j += kSampThreads) h[j] = 0ull;
    __syncthreads();
    const unsigned prefix = LEVEL == 1 ? __ldcg(&st->sel[0])
                                       : (__ldcg(&st->sel[0]) << 10) | __ldcg(&st->sel[1]);
    const int shift = LEVEL == 1 ? 10 : 0;
    const int i0 = (int)((long long)a.V * c / kChunks), i1 = (int)((long long)a.V * (c + 1) / kChunks);
    for (int base = i0; base < i1; base += kSampThreads) {   // uniform trip count
        const int i = base + (int)threadIdx.x;
        float ph = 0.0f, pl = 0.0f;
        if (i < i1) {
            ph = __ldcg(pw + 2 * i);
            pl = __ldcg(pw + 2 * i + 1);
        }
        const unsigned bits = __float_as_uint(ph);
        const bool act = i < i1 && (bits >> (shift + 10)) == prefix;
        const double pd = (double)ph + (double)pl;
        hist_add_warp(h, (bits >> shift) & (kBuckets - 1), (unsigned long long)(pd * kFix), act);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < kBuckets; j += kSampThreads)
        if (h[j]) atomicAdd(&st->hist[LEVEL][j], h[j]);
    if (!last_of_row(st, LEVEL)) return;
    const unsigned long long nf =
        (unsigned long long)(((double)__ldcg(&st->need_hi) + (double)__ldcg(&st->need_lo)) * kFix);
    pick_bucket(st, LEVEL, nf);
}

// Final pass: argmax of l (greedy) or of z + g over the nucleus; the row's
// last CTA writes the token.
__global__ void __launch_bounds__(kSampThreads) samp_pick_kernel(const SampArgs a) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y, c = blockIdx.x;
    RowState* st = row_state(a, b);
    const float* l = a.logits + (size_t)b * a.ld;
    const float* pw = row_p(a, b);
    const bool greedy = !(a.T > 0.0f);
    const bool nucleus = !greedy && a.top_p < 1.0f;
    const float tau = nucleus ? __uint_as_float(__ldcg(&st->sel[3])) : 0.0f;
    const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
    const uint64_t step = a.step_ptr ? __ldcg(reinterpret_cast<const unsigned long long*>(a.step_ptr))
                                     : a.step;
    const uint32_t s0 = (uint32_t)step, s1 = (uint32_t)(step >> 32);
    const int i0 = (int)((long long)a.V * c / kChunks), i1 = (int)((long long)a.V * (c + 1) / kChunks);
    unsigned long long best = 0ull;
    for (int i = i0 + threadIdx.x; i < i1; i += kSampThreads) {
        const float li = __ldcg(l + i);
        float v;
        if (greedy) {
            v = li;
        } else {
            if (nucleus && __ldcg(pw + 2 * i) < tau) continue;
            const uint32_t x = philox_word0((uint32_t)i, (uint32_t)b, s0, s1, k0, k1);
            const float u = ((float)(x >> 8) + 0.5f) * (1.0f / 16777216.0f);
            // z_i + g_i up to the row's constant -max / T: the same argmax
            v = __fdiv_rn(li, a.T) - logf(-logf(u));
        }
        const unsigned long long k = pack_key(v, i);
        best = k > best ? k : best;
    }
    commit_best(st, best);
    if (!last_of_row(st, 4)) return;
    if (threadIdx.x == 0) a.out[b] = (int32_t)(0xffffffffu - (unsigned)(__ldcg(&st->best) & 0xffffffffull));
}

// Advances a captured graph's step counter once the pick pass (which read
// it) has completed.
__global__ void __launch_bounds__(32) samp_step_kernel(uint64_t* step_ptr) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) *step_ptr += 1;
}

template <typename Kern>
cudaError_t launch_pass(Kern kern, int B, const SampArgs& a, const Launch& L) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kChunks, B);
    cfg.blockDim = dim3(kSampThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t sample_workspace_bytes(int B, int V) { return (size_t)B * (kStateBytes + (size_t)V * 8); }

cudaError_t launch_sample(const float* logits, int B, int V, int ld, float T, float top_p,
                          uint64_t seed, uint64_t step, float* ws, int32_t* out, const Launch& L,
                          uint64_t* step_ptr) {
    if (B <= 0) return cudaSuccess;
    SampArgs a;
    a.step_ptr = step_ptr;
    a.logits = logits;
    a.V = V;
    a.ld = ld;
    a.T = T;
    a.top_p = top_p;
    a.seed = seed;
    a.step = step;
    a.ws = reinterpret_cast<unsigned char*>(ws);
    a.out = out;
    // clear the per-row states (the p values need none)
    cudaError_t e = cudaMemsetAsync(a.ws, 0, (size_t)B * kStateBytes, L.stream);
    if (e != cudaSuccess) return e;
    const bool nucleus = T > 0.0f && top_p < 1.0f;
    if (nucleus) {
        if ((e = launch_pass(samp_max_kernel, B, a, L)) != cudaSuccess) return e;
        if ((e = launch_pass(samp_p_kernel, B, a, L)) != cudaSuccess) return e;
        if ((e = launch_pass(samp_level_kernel<1>, B, a, L)) != cudaSuccess) return e;
        if ((e = launch_pass(samp_level_kernel<2>, B, a, L)) != cudaSuccess) return e;
    }
    if ((e = launch_pass(samp_pick_kernel, B, a, L)) != cudaSuccess) return e;
    if (!step_ptr) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, samp_step_kernel, step_ptr);
}

}  // namespace a8w8
