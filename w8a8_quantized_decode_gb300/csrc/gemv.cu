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
// The streaming scheme and the arithmetic live in gemv_impl.cuh; this file
// holds the standalone kernels behind the C ABI and the layer path: the
// streaming kernel (K a multiple of 512 * k_splits, every Qwen3-14B
// projection) and a general kernel for other K (partial units masked).
#include "gemv_impl.cuh"

namespace a8w8 {

namespace {

using namespace gemv;

// Shared memory: at most 227 KB per CTA; the INT8 activation tile of a launch
// (batch tile x K bytes) gets up to 72 KB next to the weight ring.
constexpr int kMaxDynSmem = 227 * 1024;
constexpr size_t kSmemActBudget = 72 * 1024;
// Ring geometry of the streaming kernel: units per batch, batches in the ring
// (96 KB per CTA: 6 x 16 bytes per thread), batches requested before the
// dependency wait.
__host__ __device__ constexpr int ring_unr(int BT) { return BT >= 8 ? 2 : 1; }
constexpr int kRingNB = 6;
constexpr int kRingPre = 2;
// Deep form (1-2 rows): 11 batches (176 KB per CTA), all requested before
// the dependency wait. A projection whose share is at most 11 units per warp
// (O: 5120 x 5120) then has all of its weights in flight, or landed, while
// the kernel before it runs; larger ones keep the first 11 units of each
// warp's run ahead of the activation prologue.
constexpr int kDeepNB = 11;
template <int BT, int NB>
constexpr size_t stream_ring_bytes() {
    return ring_bytes<stream_threads(BT), ring_unr(BT), NB>();
}
// General kernel (any K multiple of 16).
constexpr int kGenThreads = 512;
constexpr int kGenUnroll = 8;

// ---------------------------------------------------------------------------
// Streaming kernel (K a multiple of 512 * KS).
// ---------------------------------------------------------------------------
template <int BT, int PRO, int EPI, int KS, int NB, int NBPRE>
__global__ void __launch_bounds__(stream_threads(BT), 1) gemv_stream_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    stream_gemv<BT, PRO, EPI, KS, stream_threads(BT), ring_unr(BT), NB, NBPRE>(p, smem, [] {
        pdl_wait();
        pdl_trigger();
        return true;
    });
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
    const SmemLayout L = smem_layout(BT, NSEG, KS, K, N, G, kGenThreads);
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

    if (p.clear && blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.clear_n; i += blockDim.x) p.clear[i] = 0u;
    for (int i = threadIdx.x; i < acc_n; i += blockDim.x) accs[i] = 0;
    int4 nwr[1];
    prologue<BT, PRO, 1>(p, act, xs, red, L.stage ? reinterpret_cast<bf16*>(smem + L.stage) : nullptr,
                         nwr, false, [] {});

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
    epilogue<BT, EPI, KS>(p, accs, xs, o0, nrows, rows_max, nullptr, false);
}

bool use_stream(int K, int KS) { return K % (kUnit * KS) == 0; }

template <int BT, int PRO, int EPI, int KS, int NB, int NBPRE>
cudaError_t launch_ring(const GemvParams& p, const Launch& L, bool stream) {
    auto kern = stream ? gemv_stream_kernel<BT, PRO, EPI, KS, NB, NBPRE> : gemv_kernel<BT, PRO, EPI, KS>;
    const int G = L.num_sms;
    const int nseg = EPI == EPI_SWIGLU ? 2 : 1;
    const size_t smem =
        stream ? smem_layout(BT, nseg, KS, p.K, p.N, G, stream_threads(BT), stream_ring_bytes<BT, NB>(),
                             p.late_ctas, p.late_w).total
               : smem_layout(BT, nseg, KS, p.K, p.N, G, kGenThreads).total;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(kern), [&]() -> cudaError_t {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
        });
        if (e != cudaSuccess) return e;
    }
    if (smem > (size_t)kMaxDynSmem) return cudaErrorInvalidValue;
    GemvParams q = p;
    if (!stream) q.late_ctas = 0;   // the general kernel keeps equal shares
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
    return cudaLaunchKernelEx(&cfg, kern, q);
}

template <int BT, int PRO, int EPI, int KS>
cudaError_t launch_t(const GemvParams& p, const Launch& L) {
    const bool stream = use_stream(p.K, KS);
    if constexpr (BT <= 2) {
        if (stream && p.deep) {
            const int nseg = EPI == EPI_SWIGLU ? 2 : 1;
            const size_t deep = smem_layout(BT, nseg, KS, p.K, p.N, L.num_sms, stream_threads(BT),
                                            stream_ring_bytes<BT, kDeepNB>(), p.late_ctas,
                                            p.late_w).total;
            if (deep <= (size_t)kMaxDynSmem)
                return launch_ring<BT, PRO, EPI, KS, kDeepNB, kDeepNB>(p, L, stream);
        }
    }
    return launch_ring<BT, PRO, EPI, KS, kRingNB, kRingPre>(p, L, stream);
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
