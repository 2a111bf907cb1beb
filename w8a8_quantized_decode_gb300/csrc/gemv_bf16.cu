// gemv_bf16.cu -- projections and RMSNorm of the BF16 (unquantised) decode
// layer.
//
// "perf(qwen3-a8w8): optimize decode scheduling and data paths" (pypto-lib PR
// #810; the kernel PR summary quoted there) and "Add native Qwen3 14B A8W8
// serving path" (pypto-serving PR #48), "Summary": the ordinary BF16 Qwen3-14B
// path is kept beside the A8W8 one. It is the A8W8 layer without the
// quantisation steps: y = bf16(sum_k x_k W_nk (+ residual)), one narrowing.
//
// Projection: decode-sized batches stream the BF16 weights once. The BT
// activation rows of a launch are staged in shared memory; each warp owns one
// output row at a time (for the fused Gate/Up the gate row n and the up row
// N + n) and its lanes stride over K with 16-byte weight loads, four in
// flight. Products of two BF16 values are exact in float32; each lane sums its
// share in float32 and the warp adds the lanes' sums by shuffles. The
// residual is added in float32 and the result narrowed once. The SwiGLU
// epilogue evaluates silu(g) u in two-float arithmetic from the float32 g, u.
//
// RMSNorm: one CTA per row, the sum of squares as a two-float pair, the
// normalised value narrowed once (the A8W8 layer's prologue arithmetic).
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kBfThreads = 256;
constexpr int kBfUnroll = 4;
constexpr size_t kBfSmemMax = 96 * 1024;   // staged activation rows

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 8 products of BF16 pairs added to acc (each product exact in float32).
__device__ __forceinline__ float dot8(const int4& a, const int4& b, float acc) {
    float x[8], w[8];
    unpack8(a, x);
    unpack8(b, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = __fmaf_rn(x[i], w[i], acc);
    return acc;
}

template <int BT, bool SWIGLU>
__global__ void __launch_bounds__(kBfThreads) gemv_bf16_kernel(const Bf16GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    bf16* xs = reinterpret_cast<bf16*>(smem);   // [BT][K]
    constexpr int NSEG = SWIGLU ? 2 : 1;
    const int K = p.K;
    const int nvec = K / 8;
    pdl_wait();
    for (int i = threadIdx.x; i < BT * nvec; i += kBfThreads) {
        const int m = i / nvec, c = i - m * nvec;
        int4 v = make_int4(0, 0, 0, 0);
        if (m < p.M) v = ld_cg_v4(p.x + (size_t)m * p.ldx + 8 * c);
        *reinterpret_cast<int4*>(xs + (size_t)m * K + 8 * c) = v;
    }
    __syncthreads();
    pdl_trigger();

    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (kBfThreads / 32) + (threadIdx.x >> 5);
    const int nw = gridDim.x * (kBfThreads / 32);
    for (int n = gw; n < p.N; n += nw) {
        const bf16* wr[NSEG];
        wr[0] = p.W + (size_t)n * K;
        if (SWIGLU) wr[NSEG - 1] = p.W + (size_t)(p.N + n) * K;
        float acc[NSEG][BT];
#pragma unroll
        for (int s = 0; s < NSEG; ++s)
#pragma unroll
            for (int m = 0; m < BT; ++m) acc[s][m] = 0.0f;
        int k = lane * 8;
        for (; k + (kBfUnroll - 1) * 256 < K; k += kBfUnroll * 256) {
            int4 wv[kBfUnroll][NSEG];
#pragma unroll
            for (int u = 0; u < kBfUnroll; ++u)
#pragma unroll
                for (int s = 0; s < NSEG; ++s) wv[u][s] = ld_stream_v4(wr[s] + k + 256 * u);
#pragma unroll
            for (int u = 0; u < kBfUnroll; ++u)
#pragma unroll
                for (int m = 0; m < BT; ++m) {
                    const int4 xv = *reinterpret_cast<const int4*>(xs + (size_t)m * K + k + 256 * u);
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) acc[s][m] = dot8(xv, wv[u][s], acc[s][m]);
                }
        }
        for (; k < K; k += 256) {
            int4 wv[NSEG];
#pragma unroll
            for (int s = 0; s < NSEG; ++s) wv[s] = ld_stream_v4(wr[s] + k);
#pragma unroll
            for (int m = 0; m < BT; ++m) {
                const int4 xv = *reinterpret_cast<const int4*>(xs + (size_t)m * K + k);
#pragma unroll
                for (int s = 0; s < NSEG; ++s) acc[s][m] = dot8(xv, wv[s], acc[s][m]);
            }
        }
#pragma unroll
        for (int s = 0; s < NSEG; ++s)
#pragma unroll
            for (int m = 0; m < BT; ++m) acc[s][m] = warp_sum_f(acc[s][m]);
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < BT; ++m) {
                if (m >= p.M) break;
                if (!SWIGLU) {
                    float sum = acc[0][m];
                    if (p.residual) sum = __fadd_rn(sum, bf2f(ld_cg_bf16(p.residual + (size_t)m * p.ldy + n)));
                    p.y[(size_t)m * p.ldy + n] = f2bf(sum);
                } else {
                    // silu(g) u correctly rounded (as in the A8W8 epilogue)
                    const float g = acc[0][m], u = acc[NSEG - 1][m];
                    p.y[(size_t)m * p.ldy + n] = swiglu_bf16(g, u);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kBfThreads) rmsnorm_rows_kernel(const bf16* __restrict__ x, int H,
                                                                  const bf16* __restrict__ w,
                                                                  float eps, bf16* __restrict__ y) {
    __shared__ float red[2 * (kBfThreads / 32)];
    pdl_wait();
    const int row = blockIdx.x;
    const bf16* xr = x + (size_t)row * H;
    const int nvec = H / 8;
    f2 ss = {0.0f, 0.0f};
    for (int i = threadIdx.x; i < nvec; i += kBfThreads) {
        float f[8];
        unpack8(ld_cg_v4(xr + 8 * i), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) f2_acc(ss, __fmul_rn(f[j], f[j]));
    }
    ss = warp_sum_f2(fast_two_sum(ss.hi, ss.lo));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[2 * warp] = ss.hi;
        red[2 * warp + 1] = ss.lo;
    }
    __syncthreads();
    f2 tot = {0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < kBfThreads / 32; ++i) tot = f2_add(tot, f2{red[2 * i], red[2 * i + 1]});
    const f2 inv = rms_inv(tot, H, eps);
    pdl_trigger();
    bf16* yr = y + (size_t)row * H;
    for (int i = threadIdx.x; i < nvec; i += kBfThreads) {
        float f[8], wf[8];
        unpack8(ld_cg_v4(xr + 8 * i), f);
        unpack8(ld_nc_v4(w + 8 * i), wf);
        __align__(16) bf16 o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = norm_bf16(f[j], wf[j], inv);
        *reinterpret_cast<int4*>(yr + 8 * i) = *reinterpret_cast<const int4*>(o);
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_bf(Kern kern, dim3 grid, dim3 block, size_t smem, const Launch& L,
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

template <int BT, bool SWIGLU>
cudaError_t launch_bf_t(const Bf16GemvParams& p, const Launch& L) {
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(gemv_bf16_kernel<BT, SWIGLU>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(gemv_bf16_kernel<BT, SWIGLU>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kBfSmemMax);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    const size_t smem = (size_t)BT * p.K * 2;
    if (smem > kBfSmemMax) return cudaErrorInvalidValue;
    return launch_bf(gemv_bf16_kernel<BT, SWIGLU>, dim3(2 * L.num_sms), dim3(kBfThreads), smem, L, p);
}

template <bool SWIGLU>
cudaError_t launch_bf_tile(const Bf16GemvParams& p, int bt, const Launch& L) {
    if (bt == 16) return launch_bf_t<16, SWIGLU>(p, L);
    if (bt == 8) return launch_bf_t<8, SWIGLU>(p, L);
    if (bt == 4) return launch_bf_t<4, SWIGLU>(p, L);
    if (bt == 2) return launch_bf_t<2, SWIGLU>(p, L);
    return launch_bf_t<1, SWIGLU>(p, L);
}

}  // namespace

int bf16_gemv_batch_tile(int K) {
    int bt = 16;
    while (bt > 1 && (size_t)bt * K * 2 > kBfSmemMax) bt >>= 1;
    return (size_t)K * 2 > kBfSmemMax ? 0 : bt;
}

cudaError_t launch_bf16_gemv(const Bf16GemvParams& p, bool swiglu, const Launch& L) {
    if (p.M <= 0 || p.N <= 0) return cudaSuccess;
    if (p.K <= 0 || p.K % 8 || p.ldx % 8 || L.num_sms <= 0) return cudaErrorInvalidValue;
    const int tile = bf16_gemv_batch_tile(p.K);
    if (tile == 0) return cudaErrorInvalidValue;
    for (int m0 = 0; m0 < p.M; m0 += tile) {
        Bf16GemvParams q = p;
        q.M = p.M - m0 < tile ? p.M - m0 : tile;
        q.x = p.x + (size_t)m0 * p.ldx;
        q.y = p.y + (size_t)m0 * p.ldy;
        if (p.residual) q.residual = p.residual + (size_t)m0 * p.ldy;
        int bt = 1;
        while (bt < q.M) bt <<= 1;
        cudaError_t e = swiglu ? launch_bf_tile<true>(q, bt, L) : launch_bf_tile<false>(q, bt, L);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_rmsnorm_rows(const bf16* x, int rows, int H, const bf16* w, float eps, bf16* y,
                                const Launch& L) {
    if (rows <= 0) return cudaSuccess;
    if (H <= 0 || H % 8) return cudaErrorInvalidValue;
    return launch_bf(rmsnorm_rows_kernel, dim3(rows), dim3(kBfThreads), 0, L, x, H, w, eps, y);
}

}  // namespace a8w8
