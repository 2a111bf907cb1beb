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
// halves are consecutive pieces of the same row stream, so the partials never
// leave the CTA.
//
// Design (decode, batch 1..8 rows per launch; one CTA per SM):
//   * CTA c owns output channels [c*N/G, (c+1)*N/G) (balanced to one row);
//     for the fused Gate/Up it owns the same channels of both halves. Its
//     weight rows are contiguous, so they form one byte stream (two for
//     Gate/Up) cut into 512-byte units, one 16-byte load per lane. Every warp
//     streams an equal contiguous run of units: the load pointer just advances
//     by 512 bytes per unit, with L1-bypassing 128-bit loads, double-buffered
//     (the next batch is in flight while the current one is multiplied).
//   * Row (and split) boundaries inside a run flush the warp's INT32 partial
//     sums into shared memory with an atomic add, which is exact, so how the
//     rows are split across warps does not change the result.
//   * The first batch of weight loads is issued before griddepcontrol.wait:
//     weights do not depend on the previous kernel, so under programmatic
//     dependent launch the weight stream starts while the previous kernel
//     drains.
//   * The activation rows are quantised in the prologue by every CTA
//     (redundantly, from L2): optional RMSNorm (float32, rounded to BF16),
//     absmax, then INT8 codes into shared memory. INT8 products use dp4a in
//     two independent chains.
//   * K not a multiple of 512 * k_splits falls back to a general kernel that
//     masks partial units (small shapes only).
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kUnit = 512;                // bytes per warp-wide load
constexpr int kMaxWarps = 32;
constexpr size_t kSmemActBudget = 96 * 1024;

// Streaming kernel: 4 units per batch, two batches in flight; 32 warps for
// batch tiles up to 4 rows (64 registers), 16 warps for 8-row tiles.
__host__ __device__ constexpr int stream_threads(int BT) { return BT >= 8 ? 512 : 1024; }
constexpr int kStreamUnroll = 4;
// General kernel (any K multiple of 16).
constexpr int kGenThreads = 512;
constexpr int kGenUnroll = 8;

__host__ __device__ __forceinline__ size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

template <int BT>
__device__ __forceinline__ void block_sum(float (&v)[BT], float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = warp_sum(v[b]);
        if (lane == 0) red[warp * BT + b] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = 0.0f;
        for (int w = 0; w < nw; ++w) s += red[w * BT + b];
        v[b] = s;
    }
    __syncthreads();
}

template <int BT>
__device__ __forceinline__ void block_max(float (&v)[BT], float* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = warp_max(v[b]);
        if (lane == 0) red[warp * BT + b] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        float s = 0.0f;
        for (int w = 0; w < nw; ++w) s = fmaxf(s, red[w * BT + b]);
        v[b] = s;
    }
    __syncthreads();
}

// Quantised activation rows into act[BT][K] and their scales into xs[BT].
template <int BT, int PRO>
__device__ __forceinline__ void prologue(const GemvParams& p, int8_t* act, float* xs, float* red) {
    const int K = p.K, M = p.M;
    const int nt = blockDim.x;
    if (PRO == PRO_I8) {
        const int vec = K / 16;
        for (int i = threadIdx.x; i < BT * vec; i += nt) {
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
        for (int j = threadIdx.x; j < vec; j += nt) {
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
    for (int j = threadIdx.x; j < vec; j += nt) {
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
    for (int j = threadIdx.x; j < vec; j += nt) {
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

// Dequantise in float32, add the residual or apply SwiGLU, narrow to BF16.
// accs layout: [seg][rows_max][KS][BT].
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

// Shared-memory layout common to both kernels.
struct SmemLayout {
    size_t act, accs, xs, red, total;
};
__host__ __device__ __forceinline__ SmemLayout smem_layout(int BT, int nseg, int KS, int K, int N,
                                                           int G) {
    const int rows_max = (N + G - 1) / G;
    SmemLayout s;
    s.act = 0;
    s.accs = align16((size_t)BT * K);
    s.xs = s.accs + align16((size_t)nseg * rows_max * KS * BT * 4);
    s.red = s.xs + align16((size_t)BT * 4);
    s.total = s.red + (size_t)kMaxWarps * BT * 4;
    return s;
}

// ---------------------------------------------------------------------------
// Streaming kernel (K a multiple of 512 * KS).
// ---------------------------------------------------------------------------
template <int BT, int PRO, int EPI, int KS>
__global__ void __launch_bounds__(stream_threads(BT), 1) gemv_stream_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NSEG = (EPI == EPI_SWIGLU) ? 2 : 1;
    constexpr int UNR = kStreamUnroll;
    constexpr int NW = stream_threads(BT) / 32;
    const int K = p.K, N = p.N;
    const int G = gridDim.x;
    const int o0 = (int)(((long long)N * blockIdx.x) / G);
    const int o1 = (int)(((long long)N * (blockIdx.x + 1)) / G);
    const int nrows = o1 - o0;
    const int rows_max = (N + G - 1) / G;
    const SmemLayout L = smem_layout(BT, NSEG, KS, K, N, G);
    int8_t* act = reinterpret_cast<int8_t*>(smem + L.act);
    int32_t* accs = reinterpret_cast<int32_t*>(smem + L.accs);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int upr = K / kUnit;            // units per row
    const int upp = upr / KS;             // units per piece (row split)
    const int useg = nrows * upr;         // units per segment
    const int U = NSEG * useg;
    const int u0 = (int)(((long long)U * warp) / NW);
    const int u1 = (int)(((long long)U * (warp + 1)) / NW);
    const int n = u1 - u0;

    // load stream: contiguous bytes inside a segment
    int lseg = 0, lleft = 0;
    const int8_t* lp = p.W;
    if (n > 0) {
        lseg = u0 / useg;
        const int off = u0 - lseg * useg;
        lleft = useg - off;
        lp = p.W + ((size_t)(lseg * N + o0) * K + (size_t)off * kUnit + lane * 16);
    }
    auto load_batch = [&](int4 (&dst)[UNR], int count) {
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (i < count) {
                dst[i] = ld_stream_v4(lp);
                lp += kUnit;
                if (--lleft == 0) {
                    ++lseg;
                    lleft = useg;
                    lp = p.W + ((size_t)(lseg * N + o0) * K + lane * 16);
                }
            }
        }
    };

    int4 wa[UNR], wb[UNR];
    load_batch(wa, n < UNR ? n : UNR);

    pdl_wait();
    pdl_trigger();

    const int acc_n = NSEG * rows_max * KS * BT;
    for (int i = threadIdx.x; i < acc_n; i += blockDim.x) accs[i] = 0;
    prologue<BT, PRO>(p, act, xs, red);

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
    auto compute_batch = [&](const int4 (&w)[UNR], int count) {
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (i < count) {
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
    };

    int done = 0;
    while (done < n) {
        const int ca = n - done < UNR ? n - done : UNR;
        const int rest = n - done - ca;
        const int cb = rest < UNR ? rest : UNR;
        load_batch(wb, cb);
        compute_batch(wa, ca);
        done += ca;
        if (done >= n) break;
        const int rest2 = n - done - cb;
        const int ca2 = rest2 < UNR ? rest2 : UNR;
        load_batch(wa, ca2);
        compute_batch(wb, cb);
        done += cb;
    }
    if (n > 0 && pleft != upp) flush();
    __syncthreads();
    epilogue<BT, EPI, KS>(p, accs, xs, o0, nrows, rows_max);
}

// ---------------------------------------------------------------------------
// General kernel (any K that is a multiple of 16; partial units are masked).
// ---------------------------------------------------------------------------
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

template <int BT, int KS>
__device__ __forceinline__ void flush_gen(int (&acc)[KS][BT], int32_t* accs, int seg, int r,
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

template <int BT, int PRO, int EPI, int KS>
__global__ void __launch_bounds__(kGenThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NSEG = (EPI == EPI_SWIGLU) ? 2 : 1;
    constexpr int NW = kGenThreads / 32;
    const int K = p.K, N = p.N;
    const int G = gridDim.x;
    const int o0 = (int)(((long long)N * blockIdx.x) / G);
    const int o1 = (int)(((long long)N * (blockIdx.x + 1)) / G);
    const int nrows = o1 - o0;
    const int rows_max = (N + G - 1) / G;
    const SmemLayout L = smem_layout(BT, NSEG, KS, K, N, G);
    int8_t* act = reinterpret_cast<int8_t*>(smem + L.act);
    int32_t* accs = reinterpret_cast<int32_t*>(smem + L.accs);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    const int acc_n = NSEG * rows_max * KS * BT;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int upr = (K + kUnit - 1) / kUnit;
    const int per_seg = nrows * upr;
    const int U = NSEG * per_seg;
    const int u0 = (int)((long long)U * warp / NW);
    const int u1 = (int)((long long)U * (warp + 1) / NW);
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

    int4 wv[kGenUnroll];
#pragma unroll
    for (int i = 0; i < kGenUnroll; ++i) {
        wv[i] = make_int4(0, 0, 0, 0);
        if (u0 + i < u1) {
            const int k = ld.ch * kUnit + lane_off;
            if (k < K) wv[i] = ld_stream_v4(p.W + (size_t)(ld.seg * N + o0 + ld.r) * K + k);
            advance(ld, upr, nrows);
        }
    }

    pdl_wait();
    pdl_trigger();

    for (int i = threadIdx.x; i < acc_n; i += blockDim.x) accs[i] = 0;
    prologue<BT, PRO>(p, act, xs, red);

    int acc[KS][BT];
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[s][b] = 0;
    int kseg = cur.seg, kr = cur.r;

    for (int ub = u0; ub < u1; ub += kGenUnroll) {
#pragma unroll
        for (int i = 0; i < kGenUnroll; ++i) {
            if (ub + i < u1) {
                if (cur.seg != kseg || cur.r != kr) {
                    flush_gen<BT, KS>(acc, accs, kseg, kr, rows_max, lane);
                    kseg = cur.seg;
                    kr = cur.r;
                }
                const int k = cur.ch * kUnit + lane_off;
                if (k < K) {
                    const int4 w = wv[i];
#pragma unroll
                    for (int b = 0; b < BT; ++b) {
                        const int4 a = *reinterpret_cast<const int4*>(act + (size_t)b * K + k);
                        int t = 0;
                        t = __dp4a(w.x, a.x, t);
                        t = __dp4a(w.y, a.y, t);
                        t = __dp4a(w.z, a.z, t);
                        t = __dp4a(w.w, a.w, t);
                        if (KS == 1 || k < Ks) acc[0][b] += t;
                        else acc[KS - 1][b] += t;
                    }
                }
                advance(cur, upr, nrows);
            }
        }
        if (ub + kGenUnroll < u1) {
#pragma unroll
            for (int i = 0; i < kGenUnroll; ++i) {
                if (ub + kGenUnroll + i < u1) {
                    const int k = ld.ch * kUnit + lane_off;
                    wv[i] = make_int4(0, 0, 0, 0);
                    if (k < K) wv[i] = ld_stream_v4(p.W + (size_t)(ld.seg * N + o0 + ld.r) * K + k);
                    advance(ld, upr, nrows);
                }
            }
        }
    }
    if (u0 < u1) flush_gen<BT, KS>(acc, accs, kseg, kr, rows_max, lane);
    __syncthreads();
    epilogue<BT, EPI, KS>(p, accs, xs, o0, nrows, rows_max);
}

bool use_stream(int K, int KS) { return K % (kUnit * KS) == 0; }

template <int BT, int PRO, int EPI, int KS>
cudaError_t launch_t(const GemvParams& p, const Launch& L) {
    const bool stream = use_stream(p.K, KS);
    auto kern = stream ? gemv_stream_kernel<BT, PRO, EPI, KS> : gemv_kernel<BT, PRO, EPI, KS>;
    const int G = L.num_sms;
    const int nseg = EPI == EPI_SWIGLU ? 2 : 1;
    const size_t smem = smem_layout(BT, nseg, KS, p.K, p.N, G).total;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemv_kernel<BT, PRO, EPI, KS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_stream_kernel<BT, PRO, EPI, KS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(stream ? stream_threads(BT) : kGenThreads);
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
    (void)k_splits;
    int bt = 8;
    while (bt > 1 && (size_t)bt * K > kSmemActBudget) bt >>= 1;
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
