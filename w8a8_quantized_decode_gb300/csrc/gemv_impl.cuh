// gemv_impl.cuh -- device side of the A8W8 decode projections, shared by the
// standalone projection kernels and the persistent decode-step kernel.
//
// What is computed ("perf(qwen3-a8w8): optimize decode scheduling and data
// paths", pypto-lib PR #810, "Gate/Up INT8 path" and "Decode scheduling"):
//   acc_j[m][n] = sum_{k in split j} x_q[m][k] * W[n][k]       (int32, exact)
//   p_j         = (float(acc_j) * s_x[m]) * s_w[n]              (float32)
//   y[m][n]     = bf16_rne( (p_0 [+ p_1]) [+ residual[m][n]] )
// or, for the fused Gate/Up, act = bf16_rne( silu(g) * u ) from the gate and
// up dequantised values. The two-way split-K of the down projection keeps two
// independent INT32 accumulators over the two K halves, as the pages do; the
// halves are consecutive pieces of the same row stream, so the partials never
// leave the CTA.
//
// Streaming scheme (one CTA per SM, batch tiles of 1..8 rows):
//   * CTA c owns output channels [c*N/G, (c+1)*N/G) (balanced to one row);
//     for the fused Gate/Up it owns the same channels of both halves. Its
//     weight rows are contiguous, so they form one byte stream (two for
//     Gate/Up) cut into 512-byte units, one 16-byte load per lane. Every warp
//     streams an equal contiguous run of units: the load pointer advances by
//     512 bytes per unit, each lane copying its 16 bytes into a private
//     shared-memory ring with cp.async, several batches ahead of the one
//     being multiplied.
//   * Row (and split) boundaries inside a run flush the warp's INT32 partial
//     sums into shared memory with an atomic add, which is exact, so how the
//     rows are split across warps does not change the result.
//   * The first weight batches are requested before waiting on the producer
//     of the activations (griddepcontrol.wait or a grid barrier), since
//     weights never depend on it.
//   * A prologue then quantises the activation rows (redundantly in every
//     CTA, from L2, staged once in shared memory when they fit): optional
//     RMSNorm (two-float, correctly rounded to BF16), absmax, INT8 codes into
//     shared memory; the stream multiplies with dp4a in two independent
//     chains, and a float32 dequantisation epilogue finishes.
#pragma once

#include "kernels.cuh"

namespace a8w8 {
namespace gemv {

constexpr int kUnit = 512;                // bytes per warp-wide load
constexpr int kMaxWarps = 32;

// Streaming kernel: 32 warps for batch tiles up to 4 rows (64 registers),
// 16 warps for 8-row tiles.
__host__ __device__ constexpr int stream_threads(int BT) { return BT >= 8 ? 512 : 1024; }

__host__ __device__ __forceinline__ size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Block reductions with one barrier each: every warp writes its partials,
// then every warp reads all of them (one per lane) and reduces them with
// shuffles, so each thread ends with the block result. Each call site uses
// its own region of `red`, which therefore needs no second barrier.
template <int BT>
__device__ __forceinline__ void block_max(float (&v)[BT], float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        const float s = warp_max(v[b]);
        if (lane == 0) red[b * kMaxWarps + warp] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) v[b] = warp_max(lane < nw ? red[b * kMaxWarps + lane] : 0.0f);
}

// Row sums of squares (float pairs) -> per-row RMSNorm scale 1/sqrt(ss/K+eps)
// as a float pair (see norm_bf16). red: 2 * kMaxWarps * BT floats.
template <int BT>
__device__ __forceinline__ void block_rms_inv(f2 (&ss)[BT], float* red, int K, float eps,
                                              f2 (&inv)[BT]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        const f2 t = warp_sum_f2(ss[b]);
        if (lane == 0) {
            red[2 * (b * kMaxWarps + warp)] = t.hi;
            red[2 * (b * kMaxWarps + warp) + 1] = t.lo;
        }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        f2 t = {0.0f, 0.0f};
        if (lane < nw) {
            t.hi = red[2 * (b * kMaxWarps + lane)];
            t.lo = red[2 * (b * kMaxWarps + lane) + 1];
        }
        inv[b] = rms_inv(warp_sum_f2(t), K, eps);
    }
}

// Per-thread slots of the normalisation weight held in registers (loaded
// before the dependency wait): thread t holds 8-element vectors t, t + NT, ...
// enough for K = 8192 with 1024 or 512 threads.
__host__ __device__ constexpr int norm_pre_slots(int NT) { return NT >= 1024 ? 1 : 2; }

// Row statistics with one barrier: per row the sum of squares (a float
// pair) and a maximum, reduced over the block. red: 3 * kMaxWarps * BT floats.
template <int BT>
__device__ __forceinline__ void block_stats(f2 (&ss)[BT], float (&mx)[BT], float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        const f2 t = warp_sum_f2(ss[b]);
        const float m = warp_max(mx[b]);
        if (lane == 0) {
            red[2 * (b * kMaxWarps + warp)] = t.hi;
            red[2 * (b * kMaxWarps + warp) + 1] = t.lo;
            red[2 * kMaxWarps * BT + b * kMaxWarps + warp] = m;
        }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        f2 t = {0.0f, 0.0f};
        float m = 0.0f;
        if (lane < nw) {
            t.hi = red[2 * (b * kMaxWarps + lane)];
            t.lo = red[2 * (b * kMaxWarps + lane) + 1];
            m = red[2 * kMaxWarps * BT + b * kMaxWarps + lane];
        }
        ss[b] = warp_sum_f2(t);
        mx[b] = warp_max(m);
    }
}

// The INT8 codes of eight consecutive values of one row, packed into two
// words. `fast` (the row's s > 0 with a finite R, decided once per row) takes
// quant_code's division-free form without its per-element checks; the
// results are quant_code's.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s, float R, bool fast) {
    int c[8];
    if (fast) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float q0 = __fmul_rn(f[e], R);
            const float q = __fmaf_rn(__fmaf_rn(-q0, s, f[e]), R, q0);
            c[e] = max(-127, min(127, __float2int_rn(q)));
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) c[e] = quant_code(f[e], s, R);
    }
    const unsigned lo = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    const unsigned hi = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}

// Quantised activation rows into act[BT][K] and their scales into xs[BT].
// The BF16 rows are read from L2 once (each thread issues up to four 16-byte
// loads before using any); when `stage` is given they are kept in shared
// memory for the second pass. With `nw_pre` the RMSNorm weight is taken from
// `nwr` (loaded before the wait). `issued()` is called once, right after the
// first activation loads have been issued (the caller can queue more weight
// loads behind them). With RMSNorm the stage holds the normalised BF16 rows
// afterwards.
//
// Two passes and one block reduction. Pass 1 forms each row's sum of squares
// and the maximum of |x| (plain quantisation) or of |x w| (RMSNorm). The
// second is enough for the absmax of the normalised row: x w is exact in
// float32 (two 8-bit significands), and the normalised value is the BF16
// rounding of x w times the two-float 1/rms, whose error (about 2^-47
// relative) is far below the 2^-24 gap between distinct float32 values of
// x w, so that value is a non-decreasing function of |x w| and its largest
// magnitude belongs to the largest |x w|. Pass 2 normalises (norm_bf16_fast)
// and quantises each element in one go.
template <int BT, int PRO, int NP, class Hook>
__device__ __forceinline__ void prologue(const GemvParams& p, int8_t* act, float* xs, float* red,
                                         bf16* stage, const int4 (&nwr)[NP], bool nw_pre,
                                         Hook&& issued) {
    const int K = p.K, M = p.M;
    const int nt = blockDim.x;
    if (PRO == PRO_I8) {
        issued();
        const int vec = K / 16;
        for (int i = threadIdx.x; i < BT * vec; i += nt) {
            const int b = i / vec, j = i - b * vec;
            int4 v = make_int4(0, 0, 0, 0);
            if (b < M) v = ld_cg_v4(p.xq + (size_t)b * K + 16 * j);
            *reinterpret_cast<int4*>(act + (size_t)b * K + 16 * j) = v;
        }
        if (threadIdx.x < BT) xs[threadIdx.x] = threadIdx.x < M ? __ldcg(p.x_scale + threadIdx.x) : 0.0f;
        __syncthreads();
        return;
    }
    const int vec = K / 8;
    // the RMSNorm weight of vector j: from the registers loaded before the
    // wait (slot (j - thread) / nt) or from memory
    auto norm_w = [&](int j) -> int4 {
        if (nw_pre) {
            const int slot = (j - (int)threadIdx.x) / nt;
            int4 w = make_int4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < NP; ++i)
                if (slot == i) w = nwr[i];
            return w;
        }
        return ld_nc_v4(p.norm_w + 8 * j);
    };
    // pass 1 (L2): sum of squares and max |x w| (RMSNorm) or max |x|; loads
    // in flight per row (a normalised row of K <= 8192 is one vector per
    // thread at 1024 threads, so its loads are all in flight with C = 1 or 2)
    constexpr int C = PRO == PRO_NORM_QUANT ? (BT == 1 ? 2 : 1) : (BT == 1 ? 4 : (BT == 2 ? 2 : 1));
    float mx[BT];
    f2 ss[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        mx[b] = 0.0f;
        ss[b].hi = ss[b].lo = 0.0f;
    }
    bool first = true;
    for (int j0 = threadIdx.x; j0 < vec; j0 += C * nt) {
        int4 raw[C][BT];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int j = j0 + c * nt;
#pragma unroll
            for (int b = 0; b < BT; ++b)
                raw[c][b] = (j < vec && b < M) ? ld_cg_v4(p.x + (size_t)b * p.ldx + 8 * j)
                                               : make_int4(0, 0, 0, 0);
        }
        if (first) {
            issued();
            first = false;
        }
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int j = j0 + c * nt;
            if (j < vec) {
                float w[8];
                if (PRO == PRO_NORM_QUANT) unpack8(norm_w(j), w);
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    if (b < M) {
                        if (stage) *reinterpret_cast<int4*>(stage + (size_t)b * K + 8 * j) = raw[c][b];
                        float f[8];
                        unpack8(raw[c][b], f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            if (PRO == PRO_NORM_QUANT) {
                                f2_acc(ss[b], __fmul_rn(f[e], f[e]));
                                mx[b] = fmaxf(mx[b], fabsf(__fmul_rn(f[e], w[e])));
                            } else {
                                mx[b] = fmaxf(mx[b], fabsf(f[e]));
                            }
                        }
                    }
                }
            }
        }
    }
    if (first) issued();
    float sc[BT], rc[BT];
    f2 inv[BT];
    if (PRO == PRO_NORM_QUANT) {
        block_stats<BT>(ss, mx, red);
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            inv[b] = rms_inv(ss[b], K, p.eps);
            sc[b] = __fdiv_rn(bf2f(f2_to_bf16(f2_mulf(inv[b], mx[b]))), 127.0f);
        }
    } else {
        block_max<BT>(mx, red);
#pragma unroll
        for (int b = 0; b < BT; ++b) sc[b] = __fdiv_rn(mx[b], 127.0f);
    }
    if (threadIdx.x < BT) {
#pragma unroll
        for (int b = 0; b < BT; ++b)
            if (b == (int)threadIdx.x) xs[b] = sc[b];
    }
    const bool tap = (blockIdx.x == 0) && p.tap_q != nullptr;
    const bool tapx = PRO == PRO_NORM_QUANT && (blockIdx.x == 0) && p.tap_x != nullptr;
    if (tap && threadIdx.x < M && p.tap_s) {
#pragma unroll
        for (int b = 0; b < BT; ++b)
            if (b == (int)threadIdx.x) p.tap_s[b] = sc[b];
    }
    bool fast[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        rc[b] = quant_recip(sc[b]);
        fast[b] = sc[b] != 0.0f && isfinite(rc[b]);
    }
    // pass 2: normalised BF16 values (RMSNorm) and their INT8 codes
    for (int j = threadIdx.x; j < vec; j += nt) {
        float w[8];
        if (PRO == PRO_NORM_QUANT) unpack8(norm_w(j), w);
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            uint2 code = make_uint2(0u, 0u);
            if (b < M) {
                float f[8];
                unpack8(stage ? *reinterpret_cast<const int4*>(stage + (size_t)b * K + 8 * j)
                              : ld_cg_v4(p.x + (size_t)b * p.ldx + 8 * j), f);
                if (PRO == PRO_NORM_QUANT) {
                    __align__(16) bf16 y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        y[e] = norm_bf16_fast(__fmul_rn(f[e], w[e]), inv[b]);
                        f[e] = bf2f(y[e]);
                    }
                    if (stage) *reinterpret_cast<int4*>(stage + (size_t)b * K + 8 * j) = *reinterpret_cast<const int4*>(y);
                    if (tapx) *reinterpret_cast<int4*>(p.tap_x + (size_t)b * K + 8 * j) = *reinterpret_cast<const int4*>(y);
                }
                code = quant8(f, sc[b], rc[b], fast[b]);
            }
            *reinterpret_cast<uint2*>(act + (size_t)b * K + 8 * j) = code;
            if (tap && b < M) *reinterpret_cast<uint2*>(p.tap_q + (size_t)b * K + 8 * j) = code;
        }
    }
    __syncthreads();
}

// Dequantise in float32, add the residual or apply SwiGLU, narrow to BF16.
// accs layout: [seg][rows_max][KS][BT].
// With `pre` (one element per thread), element i's weight scales and residual
// were loaded early into pre[0][i] (gate / row scale), pre[1][i] (up scale)
// and pre[2][i] (residual as float).
template <int BT, int EPI, int KS>
__device__ __forceinline__ void epilogue(const GemvParams& p, const int32_t* accs, const float* xs,
                                         int o0, int nrows, int rows_max, const float* pre,
                                         bool use_pre) {
    const int N = p.N, M = p.M;
    const int total = nrows * M;
    const int nt = blockDim.x;
    for (int i = threadIdx.x; i < total; i += nt) {
        const int b = i / nrows, r = i - b * nrows, o = o0 + r;
        if (EPI == EPI_STORE) {
            const float wsc = use_pre ? pre[i] : p.w_scale[o];
            float sum = 0.0f;
            long long full = 0;
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int a = accs[(r * KS + s) * BT + b];
                const float pj = __fmul_rn(__fmul_rn(__int2float_rn(a), xs[b]), wsc);
                sum = (s == 0) ? pj : __fadd_rn(sum, pj);
                full += a;
            }
            if (p.residual)
                sum = __fadd_rn(sum, use_pre ? pre[2 * nt + i]
                                             : bf2f(ld_cg_bf16(p.residual + (size_t)b * p.ldy + o)));
            p.y[(size_t)b * p.ldy + o] = f2bf(sum);
            if (p.acc_out) p.acc_out[(size_t)b * N + o] = (int32_t)full;
        } else {
            const int ag = accs[(0 * rows_max + r) * BT + b];
            const int au = accs[(1 * rows_max + r) * BT + b];
            const float g = __fmul_rn(__fmul_rn(__int2float_rn(ag), xs[b]),
                                      use_pre ? pre[i] : p.w_scale[o]);
            const float u = __fmul_rn(__fmul_rn(__int2float_rn(au), xs[b]),
                                      use_pre ? pre[nt + i] : p.w_scale[N + o]);
            p.y[(size_t)b * p.ldy + o] = swiglu_bf16(g, u);
            if (p.acc_out) {
                p.acc_out[(size_t)b * 2 * N + o] = ag;
                p.acc_out[(size_t)b * 2 * N + N + o] = au;
            }
        }
    }
}

// Row partition of the streaming kernel: equal shares, or with `late` > 0
// the last `late` CTAs (the ones dispatched last, onto the SMs that free up
// last) take shares of relative size w and the others the rest evenly. Each
// output row is still reduced and finished by one CTA, so where the rows run
// changes no result.
__host__ __device__ __forceinline__ bool part_skewed(int G, int late, float w) {
    return late > 0 && late < G && w > 0.0f && w < 1.0f;
}
__host__ __device__ __forceinline__ int part_bound(int N, int c, int G, int late, float w) {
    if (c <= 0) return 0;
    if (c >= G) return N;
    if (!part_skewed(G, late, w)) return (int)(((long long)N * c) / G);
    const int e = G - late;
    const float wc = c <= e ? (float)c : (float)e + (float)(c - e) * w;
    const float wg = (float)e + (float)late * w;
    return min(N, (int)((float)N * wc / wg));
}
// Rows of the largest share.
__host__ __device__ __forceinline__ int part_rows_max(int N, int G, int late, float w) {
    if (!part_skewed(G, late, w)) return (N + G - 1) / G;
    return (int)ceilf((float)N / ((float)(G - late) + (float)late * w)) + 1;
}

// Shared-memory layout common to both kernels. `stage` (BF16 copy of the
// activation rows) is present when it fits in kStageBudget (stage == 0: none).
constexpr size_t kStageBudget = 48 * 1024;
struct SmemLayout {
    size_t act, accs, xs, red, pre, stage, ring, total;
};
__host__ __device__ __forceinline__ SmemLayout smem_layout(int BT, int nseg, int KS, int K, int N,
                                                           int G, int nthreads,
                                                           size_t ring_bytes = 0, int late = 0,
                                                           float late_w = 0.0f) {
    const int rows_max = part_rows_max(N, G, late, late_w);
    SmemLayout s;
    s.act = 0;
    s.accs = align16((size_t)BT * K);
    s.xs = s.accs + align16((size_t)nseg * rows_max * KS * BT * 4);
    s.red = s.xs + align16((size_t)BT * 4);
    s.pre = align16(s.red + (size_t)3 * kMaxWarps * BT * 4);
    s.total = s.pre + (size_t)3 * nthreads * 4;
    s.stage = 0;
    if ((size_t)BT * K * 2 <= kStageBudget) {
        s.stage = s.total;
        s.total += (size_t)BT * K * 2;
    }
    s.ring = (s.total + 127) & ~size_t(127);
    s.total = s.ring + ring_bytes;
    return s;
}


// One CTA's share of a projection, streamed by NT threads. The weight units
// travel HBM -> shared memory with cp.async (no registers held while in
// flight), into a ring of NB batches of UNR units that is private to each
// lane: lane t of the CTA copies, and later reads back, only its own 16-byte
// slots, so the only synchronisation is the thread's own cp.async.wait_group.
// NBPRE batches are requested before `wait()` (griddepcontrol.wait in the
// standalone kernels, a grid barrier in the persistent step; false abandons
// the projection), the rest right behind the prologue's activation loads, so
// HBM stays busy through the dependency wait and the prologue; afterwards
// NB - 1 batches are always in flight while one is multiplied. All state
// lives in locals: the whole function is inlined into the kernel.
template <int NT, int UNR, int NB>
__host__ __device__ constexpr size_t ring_bytes() { return (size_t)NB * UNR * NT * 16; }

template <int BT, int PRO, int EPI, int KS, int NT, int UNR, int NB, int NBPRE, class Wait>
__device__ __forceinline__ bool stream_gemv(const GemvParams& p, unsigned char* smem, Wait&& wait) {
    constexpr int NSEG = (EPI == EPI_SWIGLU) ? 2 : 1;
    constexpr int NW = NT / 32;
    const int K = p.K, N = p.N;
    const int G = gridDim.x;
    const int o0 = part_bound(N, blockIdx.x, G, p.late_ctas, p.late_w);
    const int o1 = part_bound(N, blockIdx.x + 1, G, p.late_ctas, p.late_w);
    const int nrows = o1 - o0;
    const int rows_max = part_rows_max(N, G, p.late_ctas, p.late_w);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int upr = K / kUnit;            // units per row
    const int upp = upr / KS;             // units per piece (row split)
    const int useg = nrows * upr;         // units per segment
    const int U = NSEG * useg;
    const int u0 = (int)(((long long)U * warp) / NW);
    const int u1 = (int)(((long long)U * (warp + 1)) / NW);
    const int n = u1 - u0;

    const SmemLayout L = smem_layout(BT, NSEG, KS, K, N, G, NT, ring_bytes<NT, UNR, NB>(), p.late_ctas,
                                     p.late_w);
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem + L.ring) + threadIdx.x * 16u;

    // load stream: contiguous bytes inside a segment
    int lseg = 0, lleft = 0;
    const int8_t* lp = p.W;
    if (n > 0) {
        lseg = u0 / useg;
        const int off = u0 - lseg * useg;
        lleft = useg - off;
        lp = p.W + ((size_t)(lseg * N + o0) * K + (size_t)off * kUnit + lane * 16);
    }
    int issued = 0;   // units requested so far
    const uint64_t pol = l2_evict_first_policy();
    // one copy group per batch (empty when the stream is exhausted)
    auto issue_batch = [&](int slot) {
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (issued < n) {
                cp_async16_s(ring + (uint32_t)((slot * UNR + i) * NT * 16), lp, pol);
                ++issued;
                lp += kUnit;
                if (--lleft == 0) {
                    ++lseg;
                    lleft = useg;
                    lp = p.W + ((size_t)(lseg * N + o0) * K + lane * 16);
                }
            }
        }
        cp_async_commit();
    };

    // First the small operands that no kernel writes: the RMSNorm weight
    // (prologue) and this CTA's weight scales (epilogue), one epilogue element
    // per thread, so that they are not queued behind the weight stream.
    constexpr int NP = norm_pre_slots(NT);
    int4 nwr[NP];
    const int vec = K / 8;
    const bool nw_pre = PRO == PRO_NORM_QUANT && vec <= NP * NT;
    if (PRO == PRO_NORM_QUANT && nw_pre) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int j = threadIdx.x + i * NT;
            nwr[i] = j < vec ? ld_nc_v4(p.norm_w + 8 * j) : make_int4(0, 0, 0, 0);
        }
    }
    const int etotal = nrows * p.M;
    const bool ep_pre = etotal <= NT;
    const bool mine = ep_pre && (int)threadIdx.x < etotal;
    float wsg = 0.0f, wsu = 0.0f;
    if (mine) {
        const int r = (int)threadIdx.x % nrows;
        wsg = __ldg(p.w_scale + o0 + r);
        if (EPI == EPI_SWIGLU) wsu = __ldg(p.w_scale + N + o0 + r);
    }

    // then the first NBPRE batches of the ring; the others are queued behind
    // the activation loads of the prologue
#pragma unroll
    for (int b = 0; b < NBPRE; ++b) issue_batch(b);

    if (!wait()) {
        cp_async_wait_all();
        return false;
    }

    if (p.clear && blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.clear_n; i += NT) p.clear[i] = 0u;
    // the residual (written by an earlier kernel) is read right after the wait
    float resv = 0.0f;
    if (EPI == EPI_STORE && mine && p.residual) {
        const int b = (int)threadIdx.x / nrows, r = (int)threadIdx.x - b * nrows;
        resv = bf2f(ld_cg_bf16(p.residual + (size_t)b * p.ldy + o0 + r));
    }
    int8_t* act = reinterpret_cast<int8_t*>(smem + L.act);
    int32_t* accs = reinterpret_cast<int32_t*>(smem + L.accs);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    float* pre = reinterpret_cast<float*>(smem + L.pre);
    const int acc_n = NSEG * rows_max * KS * BT;
    for (int i = threadIdx.x; i < acc_n; i += blockDim.x) accs[i] = 0;
    prologue<BT, PRO, NP>(p, act, xs, red,
                          L.stage ? reinterpret_cast<bf16*>(smem + L.stage) : nullptr, nwr, nw_pre,
                          [&] {
#pragma unroll
                              for (int b = NBPRE; b < NB; ++b) issue_batch(b);
                          });
    if (mine) {   // read by the epilogue, after the barrier that ends the stream
        pre[threadIdx.x] = wsg;
        pre[NT + threadIdx.x] = wsu;
        pre[2 * NT + threadIdx.x] = resv;
    }

    // compute stream: piece = (segment, row, split)
    int cpiece = 0, pleft = 0, rleft = 0, aoff = 0;
    if (n > 0) {
        cpiece = u0 / upp;
        pleft = upp - (u0 - cpiece * upp);
        const int ju = u0 % upr;                    // unit inside the row
        rleft = upr - ju;
        aoff = ju * kUnit + lane * 16;
    }
    int acc0[BT], acc1[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) acc0[b] = acc1[b] = 0;

    auto flush = [&]() {
        // piece index -> (segment, row, split) -> shared accumulator slot
        const int split = cpiece % KS;
        const int rowg = cpiece / KS;               // segment * nrows + row
        const int seg = rowg / nrows;
        const int r = rowg - seg * nrows;
        int32_t* dst = accs + ((seg * rows_max + r) * KS + split) * BT;
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            const int v = warp_sum_i(acc0[b] + acc1[b]);
            if (lane == 0) atomicAdd(&dst[b], v);
            acc0[b] = acc1[b] = 0;
        }
    };

    int slot = 0;
    for (int done = 0; done < n; done += UNR) {
        cp_async_wait_group<NB - 1>();          // this thread's oldest batch has landed
        int4 w[UNR];
#pragma unroll
        for (int i = 0; i < UNR; ++i) w[i] = lds_v4(ring + (uint32_t)((slot * UNR + i) * NT * 16));
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (done + i < n) {
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    const int4 a = *reinterpret_cast<const int4*>(act + (size_t)b * K + aoff);
                    acc0[b] = __dp4a(w[i].x, a.x, acc0[b]);
                    acc1[b] = __dp4a(w[i].y, a.y, acc1[b]);
                    acc0[b] = __dp4a(w[i].z, a.z, acc0[b]);
                    acc1[b] = __dp4a(w[i].w, a.w, acc1[b]);
                }
                aoff += kUnit;
                if (--rleft == 0) {
                    rleft = upr;
                    aoff = lane * 16;
                }
                if (--pleft == 0) {
                    flush();
                    ++cpiece;
                    pleft = upp;
                }
            }
        }
        issue_batch(slot);                       // refill the slot just consumed
        slot = slot + 1 == NB ? 0 : slot + 1;
    }
    cp_async_wait_all();
    if (n > 0 && pleft != upp) flush();
    __syncthreads();
    epilogue<BT, EPI, KS>(p, accs, xs, o0, nrows, rows_max, pre, ep_pre);
    return true;
}

}  // namespace gemv
}  // namespace a8w8
