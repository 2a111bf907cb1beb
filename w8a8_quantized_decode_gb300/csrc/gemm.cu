// gemm.cu -- A8W8 projections of a prefill chunk (many rows): the exact INT32
// product on the tensor cores (gemm_tc.cu) and the dequantisation epilogue.
//
// Same arithmetic as gemv.cu ("perf(qwen3-a8w8): optimize decode scheduling
// and data paths", pypto-lib PR #810, "Gate/Up INT8 path"): exact INT32
// accumulators per K split, (acc * s_x) * s_w in float32, the split partials
// summed in order, the residual added, or SwiGLU of the gate and up values,
// one BF16 narrowing.
#include "gemv_impl.cuh"

namespace a8w8 {

namespace {

// Dequantisation epilogue, one thread per output: the arithmetic of the GEMV
// epilogue (gemv_impl.cuh). acc: KS planes [M][ldacc] (SwiGLU: gate columns
// [0, N), up columns [N, 2N) of one plane).
template <int EPI, int KS>
__global__ void __launch_bounds__(256) gemm_epilogue_kernel(const GemvParams p, const int32_t* acc,
                                                            int ldacc) {
    pdl_wait();
    pdl_trigger();
    if (p.clear && blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.clear_n; i += blockDim.x) p.clear[i] = 0u;
    const long total = (long)p.M * p.N;
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int b = (int)(i / p.N), o = (int)(i - (long)b * p.N);
    const float xs = __ldcg(p.x_scale + b);
    if (EPI == EPI_STORE) {
        const float wsc = p.w_scale[o];
        float sum = 0.0f;
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            const int a = acc[(size_t)s * p.M * ldacc + (size_t)b * ldacc + o];
            const float pj = __fmul_rn(__fmul_rn(__int2float_rn(a), xs), wsc);
            sum = (s == 0) ? pj : __fadd_rn(sum, pj);
        }
        if (p.residual) sum = __fadd_rn(sum, bf2f(ld_cg_bf16(p.residual + (size_t)b * p.ldy + o)));
        p.y[(size_t)b * p.ldy + o] = f2bf(sum);
    } else {
        const int ag = acc[(size_t)b * ldacc + o];
        const int au = acc[(size_t)b * ldacc + p.N + o];
        const float gv = __fmul_rn(__fmul_rn(__int2float_rn(ag), xs), p.w_scale[o]);
        const float uv = __fmul_rn(__fmul_rn(__int2float_rn(au), xs), p.w_scale[p.N + o]);
        p.y[(size_t)b * p.ldy + o] = swiglu_bf16(gv, uv);
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, const Launch& L,
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

}  // namespace

bool gemm_supported(int K, int k_splits) { return gemm_tc_supported(K, k_splits); }

size_t gemm_acc_bytes(int M, int N, int epilogue, int k_splits) {
    const size_t cols = (size_t)(epilogue == EPI_SWIGLU ? 2 * N : N);
    return (size_t)k_splits * M * cols * 4;
}

cudaError_t launch_gemm_projection(int epilogue, int k_splits, const GemvParams& p, int32_t* acc,
                                   uint16_t* x16, const Launch& L) {
    if (p.M <= 0) return cudaSuccess;
    if (!p.xq || !p.x_scale || !x16 || !gemm_supported(p.K, k_splits)) return cudaErrorInvalidValue;
    {
        cudaError_t e = launch_i8_to_f16(p.xq, (size_t)p.M * p.K, x16, L);
        if (e != cudaSuccess) return e;
    }
    if (epilogue == EPI_SWIGLU && k_splits != 1) return cudaErrorInvalidValue;
    const int Nc = epilogue == EPI_SWIGLU ? 2 * p.N : p.N;
    const int Ks = p.K / k_splits;
    for (int s = 0; s < k_splits; ++s) {
        cudaError_t e = launch_gemm_tc(x16, p.M, p.W, Nc, p.K, s * Ks, (s + 1) * Ks,
                                       acc + (size_t)s * p.M * Nc, Nc, p.err, L);
        if (e != cudaSuccess) return e;
    }
    const long total = (long)p.M * p.N;
    const dim3 eg((unsigned)((total + 255) / 256));
    if (epilogue == EPI_SWIGLU)
        return launch_pdl(gemm_epilogue_kernel<EPI_SWIGLU, 1>, eg, dim3(256), 0, L, p,
                          (const int32_t*)acc, Nc);
    if (k_splits == 2)
        return launch_pdl(gemm_epilogue_kernel<EPI_STORE, 2>, eg, dim3(256), 0, L, p,
                          (const int32_t*)acc, Nc);
    return launch_pdl(gemm_epilogue_kernel<EPI_STORE, 1>, eg, dim3(256), 0, L, p,
                      (const int32_t*)acc, Nc);
}

}  // namespace a8w8
