// gemv.cu -- A8W8 decode projections as HBM-streaming INT8 GEMV (dp4a).
//
// What is computed ("perf(qwen3-a8w8): optimize decode scheduling and data
// paths", pypto-lib PR #810, "Gate/Up INT8 path" and "Decode scheduling"):
//   acc_j[m][n] = sum_{k in split j} x_q[m][k] * W[n][k]       (int32, exact)
//   p_j         = (float(acc_j) * s_x[m]) * s_w[n]              (float32)
//   y[m][n]     = bf16_rne( (p_0 [+ p_1]) [+ residual[m][n]] )
// or, for the fused Gate/Up, act = bf16_rne( silu(g) * u ) from the gate and
// up dequantised values. The two-way split-K of the down projection keeps two
// independent INT32 accumulators over the two K halves, as the pages do; the
// halves stay inside one warp because the 5120 output rows already give every
// SM enough independent rows, so the partials never leave registers.
//
// Design (decode, batch 1..8 rows per launch):
//   * One CTA per SM, 16 warps. CTA c owns output channels [c*N/G, (c+1)*N/G)
//     (balanced to one row). The CTA's weight bytes are cut into 512-byte
//     units (one 16-byte load per lane) and every warp streams an equal,
//     contiguous run of units with 128-bit L1-bypassing loads, kUnroll units
//     in flight per warp (64 KB per SM). Row boundaries inside a run flush
//     the warp's INT32 partial sums into shared memory with an atomic add,
//     which is exact, so the split of rows across warps does not change the
//     result.
//   * The first batch of weight loads is issued before griddepcontrol.wait:
//     weights do not depend on the previous kernel, so with programmatic
//     dependent launch the weight stream starts while the previous kernel
//     drains.
//   * The activation rows are quantised in the prologue by every CTA
//     (redundantly, from L2): optional RMSNorm (float32, rounded to BF16),
//     absmax, then INT8 codes into shared memory. INT8 x INT8 products run on
//     dp4a with the activation read from shared memory.
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnit = 512;      // bytes per warp-wide load
constexpr int kUnroll = 8;
constexpr size_t kSmemActBudget = 96 * 1024;

__host__ __device__ __forceinline__ size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

struct Cursor {
    int seg, r, ch;
};

__device__ __forceinline__ void advance(Cursor& c, int upr, int nrows) {
    if (++c.ch == upr) {
        c.ch = 0;
        if (++c.r == nrows) {
            c.r = 0;
            ++c.seg;
        }
    }
}

template <int BT>
__device__ __forceinline__ void block_sum(float (&v)[BT], float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = warp_sum(v[b]);
        if (lane == 0) red[warp * BT + b] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w * BT + b];
        v[b] = s;
    }
    __syncthreads();
}

template <int BT>
__device__ __forceinline__ void block_max(float (&v)[BT], float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = warp_max(v[b]);
        if (lane == 0) red[warp * BT + b] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s = fmaxf(s, red[w * BT + b]);
        v[b] = s;
    }
    __syncthreads();
}

// Quantised activation rows into act[BT][K] and their scales into xs[BT].
template <int BT, int PRO>
__device__ __forceinline__ void prologue(const GemvParams& p, int8_t* act, float* xs, float* red) {
    const int K = p.K, M = p.M;
    if (PRO == PRO_I8) {
        const int vec = K / 16;
        for (int i = threadIdx.x; i < BT * vec; i += kThreads) {
            const int b = i / vec, j = i - b * vec;
            int4 v = make_int4(0, 0, 0, 0);
            if (b < M) v = ld_nc_v4(p.xq + (size_t)b * K + 16 * j);
            *reinterpret_cast<int4*>(act + (size_t)b * K + 16 * j) = v;
        }
        if (threadIdx.x < BT) xs[threadIdx.x] = threadIdx.x < M ? p.x_scale[threadIdx.x] : 0.0f;
        __syncthreads();
        return;
    }
    const int vec = K / 8;
    float inv[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) inv[b] = 1.0f;
    if (PRO == PRO_NORM_QUANT) {
        float ss[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) ss[b] = 0.0f;
        for (int j = threadIdx.x; j < vec; j += kThreads) {
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                if (b < M) {
                    float f[8];
                    unpack8(ld_nc_v4(p.x + (size_t)b * p.ldx + 8 * j), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss[b] += f[e] * f[e];
                }
            }
        }
        block_sum<BT>(ss, red);
#pragma unroll
        for (int b = 0; b < BT; ++b)
            inv[b] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss[b], (float)K), p.eps)));
    }
    // absmax of the BF16 row that is quantised
    float am[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) am[b] = 0.0f;
    for (int j = threadIdx.x; j < vec; j += kThreads) {
        float w[8];
        if (PRO == PRO_NORM_QUANT) unpack8(ld_nc_v4(p.norm_w + 8 * j), w);
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            if (b < M) {
                float f[8];
                unpack8(ld_nc_v4(p.x + (size_t)b * p.ldx + 8 * j), f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float y = f[e];
                    if (PRO == PRO_NORM_QUANT) y = bf2f(f2bf(__fmul_rn(__fmul_rn(y, inv[b]), w[e])));
                    am[b] = fmaxf(am[b], fabsf(y));
                }
            }
        }
    }
    block_max<BT>(am, red);
    float sc[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) sc[b] = __fdiv_rn(am[b], 127.0f);
    if (threadIdx.x < BT) {
#pragma unroll
        for (int b = 0; b < BT; ++b)
            if (b == (int)threadIdx.x) xs[b] = sc[b];
    }
    const bool tap = (blockIdx.x == 0) && p.tap_q != nullptr;
    const bool tapx = (blockIdx.x == 0) && p.tap_x != nullptr && PRO == PRO_NORM_QUANT;
    if (tap && threadIdx.x < M && p.tap_s) {
#pragma unroll
        for (int b = 0; b < BT; ++b)
            if (b == (int)threadIdx.x) p.tap_s[b] = sc[b];
    }
    for (int j = threadIdx.x; j < vec; j += kThreads) {
        float w[8];
        if (PRO == PRO_NORM_QUANT) unpack8(ld_nc_v4(p.norm_w + 8 * j), w);
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            uint32_t lo = 0, hi = 0;
            if (b < M) {
                float f[8];
                unpack8(ld_nc_v4(p.x + (size_t)b * p.ldx + 8 * j), f);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float y = f[e];
                    if (PRO == PRO_NORM_QUANT) {
                        const bf16 yb = f2bf(__fmul_rn(__fmul_rn(y, inv[b]), w[e]));
                        if (tapx) p.tap_x[(size_t)b * K + 8 * j + e] = yb;
                        y = bf2f(yb);
                    }
                    const uint32_t c = (uint32_t)(quant_code(y, sc[b]) & 0xff);
                    if (e < 4) lo |= c << (8 * e);
                    else hi |= c << (8 * (e - 4));
                }
            }
            *reinterpret_cast<uint2*>(act + (size_t)b * K + 8 * j) = make_uint2(lo, hi);
            if (tap && b < M) *reinterpret_cast<uint2*>(p.tap_q + (size_t)b * K + 8 * j) = make_uint2(lo, hi);
        }
    }
    __syncthreads();
}

template <int BT, int KS>
__device__ __forceinline__ void flush(int (&acc)[KS][BT], int32_t* accs, int seg, int r,
                                      int rows_max, int lane) {
#pragma unroll
    for (int s = 0; s < KS; ++s) {
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            const int v = warp_sum_i(acc[s][b]);
            if (lane == 0) atomicAdd(&accs[((seg * rows_max + r) * KS + s) * BT + b], v);
            acc[s][b] = 0;
        }
    }
}

// Dequantise in float32, add the residual or apply SwiGLU, narrow to BF16.
template <int BT, int EPI, int KS>
__device__ __forceinline__ void epilogue(const GemvParams& p, const int32_t* accs, const float* xs,
                                         int o0, int nrows, int rows_max) {
    const int N = p.N, M = p.M;
    const int total = nrows * M;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int b = i / nrows, r = i - b * nrows, o = o0 + r;
        if (EPI == EPI_STORE) {
            float sum = 0.0f;
            long long full = 0;
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int a = accs[(r * KS + s) * BT + b];
                const float pj = __fmul_rn(__fmul_rn(__int2float_rn(a), xs[b]), p.w_scale[o]);
                sum = (s == 0) ? pj : __fadd_rn(sum, pj);
                full += a;
            }
            if (p.residual) sum = __fadd_rn(sum, bf2f(p.residual[(size_t)b * p.ldy + o]));
            p.y[(size_t)b * p.ldy + o] = f2bf(sum);
            if (p.acc_out) p.acc_out[(size_t)b * N + o] = (int32_t)full;
        } else {
            const int ag = accs[(0 * rows_max + r) * BT + b];
            const int au = accs[(1 * rows_max + r) * BT + b];
            const float g = __fmul_rn(__fmul_rn(__int2float_rn(ag), xs[b]), p.w_scale[o]);
            const float u = __fmul_rn(__fmul_rn(__int2float_rn(au), xs[b]), p.w_scale[N + o]);
            // silu(g) = g * sigmoid(g), with exp taken of -|g| so that it never overflows
            const float e = expf(-fabsf(g));
            const float sig = g >= 0.0f ? __fdiv_rn(1.0f, __fadd_rn(1.0f, e))
                                        : __fdiv_rn(e, __fadd_rn(1.0f, e));
            const float si = __fmul_rn(g, sig);
            p.y[(size_t)b * p.ldy + o] = f2bf(__fmul_rn(si, u));
            if (p.acc_out) {
                p.acc_out[(size_t)b * 2 * N + o] = ag;
                p.acc_out[(size_t)b * 2 * N + N + o] = au;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Streaming through shared memory with the bulk-copy (TMA) engine, for
// K a multiple of 512 * k_splits (every Qwen3-14B projection). The CTA's rows
// are cut into stages of whole rows (about 20 KB) held in a ring of
// `stages` buffers (about 120 KB). Thread 0 issues one bulk copy per stage;
// the first ring-full is issued before griddepcontrol.wait, so the weights of
// this projection stream in while the previous kernel finishes. Consumers
// (all 16 warps) split each stage into 512-byte units (16 bytes per lane),
// accumulate dp4a partial sums and merge rows with shared-memory INT32
// atomics; after a stage every warp arrives on its "empty" barrier and thread
// 0 refills it with the stage `stages` ahead.
// ---------------------------------------------------------------------------
struct TmaPlan {
    int rows_per_stage;
    int stages;
    size_t stage_bytes;
};

constexpr size_t kStageTarget = 20 * 1024;
constexpr size_t kRingTarget = 120 * 1024;
constexpr int kMaxStages = 8;

__host__ __device__ __forceinline__ TmaPlan tma_plan(int K) {
    TmaPlan t;
    t.rows_per_stage = (int)(kStageTarget / (size_t)K);
    if (t.rows_per_stage < 1) t.rows_per_stage = 1;
    t.stage_bytes = (size_t)t.rows_per_stage * K;
    t.stages = (int)(kRingTarget / t.stage_bytes);
    if (t.stages > kMaxStages) t.stages = kMaxStages;
    if (t.stages < 2) t.stages = 2;
    return t;
}

template <int BT, int PRO, int EPI, int KS>
__global__ void __launch_bounds__(kThreads, 1) gemv_tma_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NSEG = (EPI == EPI_SWIGLU) ? 2 : 1;
    const int K = p.K, N = p.N;
    const int G = gridDim.x;
    const int o0 = (int)(((long long)N * blockIdx.x) / G);
    const int o1 = (int)(((long long)N * (blockIdx.x + 1)) / G);
    const int nrows = o1 - o0;
    const int rows_max = (N + G - 1) / G;
    const TmaPlan plan = tma_plan(K);
    const int R = plan.rows_per_stage, NS = plan.stages;
    unsigned char* ring = smem;
    int8_t* act = reinterpret_cast<int8_t*>(smem + plan.stage_bytes * NS);
    int32_t* accs = reinterpret_cast<int32_t*>(smem + plan.stage_bytes * NS + align16((size_t)BT * K));
    const int acc_n = NSEG * rows_max * KS * BT;
    float* xs = reinterpret_cast<float*>(accs + acc_n);
    float* red = xs + BT;
    uint64_t* full = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(red + kWarps * BT) + 7) & ~uintptr_t(7));
    uint64_t* empty = full + NS;
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int upr = K / kUnit;                 // units per row
    const int per_seg = (nrows + R - 1) / R;   // stages per segment
    const int C = NSEG * per_seg;              // stages in total
    const int Ks_units = upr / KS;             // units per K split

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    uint64_t policy = 0;
    int issued = 0;   // stages issued so far (thread 0 only)
    auto issue = [&](int c) {
        ++issued;
        const int seg = c / per_seg;
        const int rf = (c - seg * per_seg) * R;
        const int rows = min(R, nrows - rf);
        const unsigned bytes = (unsigned)(rows * K);
        const int s = c % NS;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(ring + (size_t)s * plan.stage_bytes, p.W + (size_t)(seg * N + o0 + rf) * K, bytes,
                 &full[s], policy);
    };
    if (threadIdx.x == 0) {
        policy = l2_evict_first_policy();
        const int first = C < NS ? C : NS;
        for (int c = 0; c < first; ++c) issue(c);
    }

    pdl_wait();
    pdl_trigger();

    for (int i = threadIdx.x; i < acc_n; i += kThreads) accs[i] = 0;
    prologue<BT, PRO>(p, act, xs, red);

    int acc[KS][BT];
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[s][b] = 0;

    bool ok = true;
    for (int c = 0; c < C; ++c) {
        const int s = c % NS;
        const unsigned par = (unsigned)((c / NS) & 1);
        if (!mbar_wait(&full[s], par)) {
            ok = false;
            break;
        }
        const int seg = c / per_seg;
        const int rf = (c - seg * per_seg) * R;
        const int rows = min(R, nrows - rf);
        const int U = rows * upr;
        const int u0 = (U * warp) / kWarps, u1 = (U * (warp + 1)) / kWarps;
        if (u0 < u1) {
            int r = u0 / upr, j = u0 - r * upr;
            int kr = r;
            const unsigned char* stage = ring + (size_t)s * plan.stage_bytes;
            for (int u = u0; u < u1; ++u) {
                if (r != kr) {
                    flush<BT, KS>(acc, accs, seg, rf + kr, rows_max, lane);
                    kr = r;
                }
                const int4 w = *reinterpret_cast<const int4*>(stage + (size_t)r * K + j * kUnit + lane * 16);
                const int k = j * kUnit + lane * 16;
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    const int4 a = *reinterpret_cast<const int4*>(act + (size_t)b * K + k);
                    int t = 0;
                    t = __dp4a(w.x, a.x, t);
                    t = __dp4a(w.y, a.y, t);
                    t = __dp4a(w.z, a.z, t);
                    t = __dp4a(w.w, a.w, t);
                    if (KS == 1 || j < Ks_units) acc[0][b] += t;
                    else acc[KS - 1][b] += t;
                }
                if (++j == upr) {
                    j = 0;
                    ++r;
                }
            }
            flush<BT, KS>(acc, accs, seg, rf + kr, rows_max, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (threadIdx.x == 0 && c + NS < C) {
            if (mbar_wait(&empty[s], par)) {
                issue(c + NS);
            } else {
                ok = false;
            }
        }
        __syncwarp();
        if (!ok || s_abort) break;
    }
    if (!ok) {
        s_abort = 1;
        set_error(p.err, 0x20u);
    }
    __syncthreads();
    if (s_abort) {
        // let every issued copy land before the CTA's shared memory is released
        if (threadIdx.x == 0) {
            for (int c = issued - NS < 0 ? 0 : issued - NS; c < issued; ++c)
                (void)mbar_wait(&full[c % NS], (unsigned)((c / NS) & 1));
        }
        __syncthreads();
        return;
    }
    epilogue<BT, EPI, KS>(p, accs, xs, o0, nrows, rows_max);
}

template <int BT, int PRO, int EPI, int KS>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NSEG = (EPI == EPI_SWIGLU) ? 2 : 1;
    const int K = p.K, N = p.N;
    const int G = gridDim.x;
    const int o0 = (int)(((long long)N * blockIdx.x) / G);
    const int o1 = (int)(((long long)N * (blockIdx.x + 1)) / G);
    const int nrows = o1 - o0;
    const int rows_max = (N + G - 1) / G;
    int8_t* act = reinterpret_cast<int8_t*>(smem);
    int32_t* accs = reinterpret_cast<int32_t*>(smem + align16((size_t)BT * K));
    const int acc_n = NSEG * rows_max * KS * BT;
    float* xs = reinterpret_cast<float*>(accs + acc_n);
    float* red = xs + BT;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int upr = (K + kUnit - 1) / kUnit;
    const int per_seg = nrows * upr;
    const int U = NSEG * per_seg;
    const int u0 = (int)((long long)U * warp / kWarps);
    const int u1 = (int)((long long)U * (warp + 1) / kWarps);
    const int Ks = K / KS;
    const int lane_off = lane * 16;

    Cursor ld;
    ld.seg = per_seg ? u0 / per_seg : 0;
    {
        const int rem = per_seg ? u0 - ld.seg * per_seg : 0;
        ld.r = rem / upr;
        ld.ch = rem - ld.r * upr;
    }
    Cursor cur = ld;

    int4 wv[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        wv[i] = make_int4(0, 0, 0, 0);
        if (u0 + i < u1) {
            const int k = ld.ch * kUnit + lane_off;
            if (k < K) wv[i] = ld_stream_v4(p.W + (size_t)(ld.seg * N + o0 + ld.r) * K + k);
            advance(ld, upr, nrows);
        }
    }

    pdl_wait();
    pdl_trigger();

    for (int i = threadIdx.x; i < acc_n; i += kThreads) accs[i] = 0;
    prologue<BT, PRO>(p, act, xs, red);

    int acc[KS][BT];
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[s][b] = 0;
    int kseg = cur.seg, kr = cur.r;

    for (int ub = u0; ub < u1; ub += kUnroll) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            if (ub + i < u1) {
                if (cur.seg != kseg || cur.r != kr) {
                    flush<BT, KS>(acc, accs, kseg, kr, rows_max, lane);
                    kseg = cur.seg;
                    kr = cur.r;
                }
                const int k = cur.ch * kUnit + lane_off;
                if (k < K) {
                    const int4 w = wv[i];
#pragma unroll
                    for (int b = 0; b < BT; ++b) {
                        const int4 a = *reinterpret_cast<const int4*>(act + (size_t)b * K + k);
                        if (KS == 1) {
                            int t = acc[0][b];
                            t = __dp4a(w.x, a.x, t);
                            t = __dp4a(w.y, a.y, t);
                            t = __dp4a(w.z, a.z, t);
                            t = __dp4a(w.w, a.w, t);
                            acc[0][b] = t;
                        } else {
                            int t = 0;
                            t = __dp4a(w.x, a.x, t);
                            t = __dp4a(w.y, a.y, t);
                            t = __dp4a(w.z, a.z, t);
                            t = __dp4a(w.w, a.w, t);
                            if (k < Ks) acc[0][b] += t;
                            else acc[KS - 1][b] += t;
                        }
                    }
                }
                advance(cur, upr, nrows);
            }
        }
        if (ub + kUnroll < u1) {
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                if (ub + kUnroll + i < u1) {
                    const int k = ld.ch * kUnit + lane_off;
                    wv[i] = make_int4(0, 0, 0, 0);
                    if (k < K) wv[i] = ld_stream_v4(p.W + (size_t)(ld.seg * N + o0 + ld.r) * K + k);
                    advance(ld, upr, nrows);
                }
            }
        }
    }
    if (u0 < u1) flush<BT, KS>(acc, accs, kseg, kr, rows_max, lane);
    __syncthreads();

    epilogue<BT, EPI, KS>(p, accs, xs, o0, nrows, rows_max);
}

size_t gemv_smem_bytes(int BT, int nseg, int KS, int K, int N, int G) {
    const int rows_max = (N + G - 1) / G;
    return align16((size_t)BT * K) + (size_t)nseg * rows_max * KS * BT * 4 + (size_t)BT * 4 +
           (size_t)kWarps * BT * 4;
}

bool use_tma(int K, int KS) { return K % (kUnit * KS) == 0; }

size_t gemv_tma_smem_bytes(int BT, int nseg, int KS, int K, int N, int G) {
    const TmaPlan t = tma_plan(K);
    return t.stage_bytes * t.stages + gemv_smem_bytes(BT, nseg, KS, K, N, G) + 8 + 16 * t.stages;
}

template <int BT, int PRO, int EPI, int KS>
cudaError_t launch_t(const GemvParams& p, const Launch& L) {
    const bool tma = use_tma(p.K, KS);
    auto kern = tma ? gemv_tma_kernel<BT, PRO, EPI, KS> : gemv_kernel<BT, PRO, EPI, KS>;
    const int G = L.num_sms;
    const int nseg = EPI == EPI_SWIGLU ? 2 : 1;
    const size_t smem = tma ? gemv_tma_smem_bytes(BT, nseg, KS, p.K, p.N, G)
                            : gemv_smem_bytes(BT, nseg, KS, p.K, p.N, G);
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<BT, PRO, EPI, KS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_tma_kernel<BT, PRO, EPI, KS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    if (smem > 220 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int PRO, int EPI, int KS>
cudaError_t launch_bt(const GemvParams& p, const Launch& L) {
    if (p.M <= 1) return launch_t<1, PRO, EPI, KS>(p, L);
    if (p.M <= 2) return launch_t<2, PRO, EPI, KS>(p, L);
    if (p.M <= 4) return launch_t<4, PRO, EPI, KS>(p, L);
    return launch_t<8, PRO, EPI, KS>(p, L);
}

}  // namespace

int gemv_max_batch_tile(int K, int k_splits) {
    const size_t budget = use_tma(K, k_splits)
                              ? 200 * 1024 - tma_plan(K).stage_bytes * tma_plan(K).stages
                              : kSmemActBudget;
    int bt = 8;
    while (bt > 1 && (size_t)bt * K > budget) bt >>= 1;
    return bt;
}

cudaError_t launch_gemv(int prologue, int epilogue, int k_splits, const GemvParams& p,
                        const Launch& L) {
    if (p.M <= 0) return cudaSuccess;
    if (p.M > gemv_max_batch_tile(p.K, k_splits)) return cudaErrorInvalidValue;
    if (epilogue == EPI_STORE) {
        if (k_splits == 1) {
            if (prologue == PRO_I8) return launch_bt<PRO_I8, EPI_STORE, 1>(p, L);
            if (prologue == PRO_QUANT) return launch_bt<PRO_QUANT, EPI_STORE, 1>(p, L);
            return launch_bt<PRO_NORM_QUANT, EPI_STORE, 1>(p, L);
        }
        if (k_splits == 2) {
            if (prologue == PRO_I8) return launch_bt<PRO_I8, EPI_STORE, 2>(p, L);
            if (prologue == PRO_QUANT) return launch_bt<PRO_QUANT, EPI_STORE, 2>(p, L);
        }
        return cudaErrorInvalidValue;
    }
    if (k_splits != 1) return cudaErrorInvalidValue;
    if (prologue == PRO_I8) return launch_bt<PRO_I8, EPI_SWIGLU, 1>(p, L);
    if (prologue == PRO_NORM_QUANT) return launch_bt<PRO_NORM_QUANT, EPI_SWIGLU, 1>(p, L);
    return cudaErrorInvalidValue;
}

}  // namespace a8w8
