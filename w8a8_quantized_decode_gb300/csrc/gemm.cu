// gemm.cu -- A8W8 projections of a prefill chunk (many rows): a tiled GEMM on
// the tensor cores with an exact INT32 result, and the dequantisation epilogue.
//
// Same arithmetic as gemv.cu ("perf(qwen3-a8w8): optimize decode scheduling
// and data paths", pypto-lib PR #810, "Gate/Up INT8 path"): exact INT32
// accumulators per K split, (acc * s_x) * s_w in float32, the split partials
// summed in order, the residual added, or SwiGLU of the gate and up values,
// one BF16 narrowing.
//
// GEMM: C[m][n] = sum_{k in [k0, k1)} A[m][k] * W[n][k], A the INT8 activation
// codes [M, K], W the INT8 weights [N, K]. One CTA of 256 threads computes a
// 128 x 128 tile of C over 64-column K steps:
//   * the INT8 tiles of A and W are copied with cp.async into a two-stage
//     shared-memory buffer, one step ahead of the one in use;
//   * each step's tiles are converted once to FP16 (exact: |codes| <= 128)
//     into padded shared tiles, and the 8 warps (2 x 4, warp tile 64 x 32)
//     run mma.sync m16n8k16 from ldmatrix fragments with FP32 accumulators;
//   * every product is an integer below 2^15, and 16 steps (1024 columns) sum
//     to below 2^24 in magnitude, where float32 holds every integer: the
//     accumulators are exact; they are converted to INT32 and added into an
//     INT32 tile in shared memory every 16 steps, which is written out at the
//     end.
#include <cstdlib>

#include "gemv_impl.cuh"

namespace a8w8 {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kGemmThreads = 256;
constexpr int kChunkSteps = 16;          // steps per exact float32 chunk
constexpr int kHP = kBK + 8;             // FP16 tile row pitch (halves)
constexpr int kCP = kBN + 4;             // INT32 tile row pitch (words): the 8 rows
                                         // a flush instruction touches fall in 8 bank groups

struct GemmSmem {
    size_t a8, b8, ah, bh, c, total;
};
__host__ __device__ inline GemmSmem gemm_smem() {
    GemmSmem s;
    s.a8 = 0;                                        // [2][BM][BK] int8
    s.b8 = s.a8 + (size_t)2 * kBM * kBK;             // [2][BN][BK] int8
    s.ah = s.b8 + (size_t)2 * kBN * kBK;             // [BM][kHP] f16
    s.bh = s.ah + (size_t)kBM * kHP * 2;             // [BN][kHP] f16
    s.c = s.bh + (size_t)kBN * kHP * 2;              // [BM][kCP] int32
    s.total = s.c + (size_t)kBM * kCP * 4;
    return s;
}

// 4 INT8 -> 2 x f16x2 (exact): byte v becomes the f16 1024 + (v + 128),
// then 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 lf = __hsub2(*reinterpret_cast<const __half2*>(&l), off);
    const __half2 hf = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
    lo = *reinterpret_cast<const uint32_t*>(&lf);
    hi = *reinterpret_cast<const uint32_t*>(&hf);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16_z(uint32_t s, const void* g, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(g), "r"(src_bytes)
                 : "memory");
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_i8_kernel(const int8_t* __restrict__ A, int lda, const int8_t* __restrict__ W, int ldw,
                   int M, int N, int k0, int k1, int32_t* __restrict__ C, int ldc) {
    extern __shared__ __align__(16) unsigned char smem[];
    const GemmSmem L = gemm_smem();
    int8_t* a8 = reinterpret_cast<int8_t*>(smem + L.a8);
    int8_t* b8 = reinterpret_cast<int8_t*>(smem + L.b8);
    __half* ah = reinterpret_cast<__half*>(smem + L.ah);
    __half* bh = reinterpret_cast<__half*>(smem + L.bh);
    int32_t* sc = reinterpret_cast<int32_t*>(smem + L.c);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    // M tiles vary fastest: the CTAs that share a weight tile run together and
    // read it from L2 after the first
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
    const int wm = warp >> 2, wn = warp & 3;     // warp tile rows wm*64, cols wn*32
    const int steps = (k1 - k0) / kBK;

    pdl_wait();
    pdl_trigger();

    for (int i = tid; i < kBM * kCP; i += kGemmThreads) sc[i] = 0;

    // copies of step s into stage s & 1: 512 16-byte pieces per operand, 2 per thread
    auto issue = [&](int s) {
        const int kk = k0 + s * kBK;
        const int st = s & 1;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = tid + i * kGemmThreads;
            const int row = c >> 2, col = (c & 3) * 16;
            const bool okA = m0 + row < M, okB = n0 + row < N;
            const int8_t* srcA = okA ? A + (size_t)(m0 + row) * lda + kk + col : A;
            const int8_t* srcB = okB ? W + (size_t)(n0 + row) * ldw + kk + col : W;
            cp_async16_z((uint32_t)__cvta_generic_to_shared(a8 + (size_t)(st * kBM + row) * kBK + col),
                         srcA, okA ? 16 : 0);
            cp_async16_z((uint32_t)__cvta_generic_to_shared(b8 + (size_t)(st * kBN + row) * kBK + col),
                         srcB, okB ? 16 : 0);
        }
        cp_async_commit();
    };

    float acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.0f;

    // ldmatrix lane addresses: A (m16 x k16 per x4), B (two n8 tiles x k16 per x4)
    const int lrow = lane & 7, lsel = lane >> 3;
    const uint32_t ah_base = (uint32_t)__cvta_generic_to_shared(ah);
    const uint32_t bh_base = (uint32_t)__cvta_generic_to_shared(bh);
    const uint32_t a_lane = ah_base + (uint32_t)(((wm * 64 + lrow + 8 * (lsel & 1)) * kHP + 8 * (lsel >> 1)) * 2);
    const uint32_t b_lane = bh_base + (uint32_t)(((wn * 32 + lrow + 8 * (lsel >> 1)) * kHP + 8 * (lsel & 1)) * 2);

    if (steps > 0) issue(0);
    for (int s = 0; s < steps; ++s) {
        if (s + 1 < steps) {
            issue(s + 1);
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();   // step s landed; the FP16 tiles are free
        {
            const int st = s & 1;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = tid + i * kGemmThreads;
                const int row = c >> 2, col = (c & 3) * 16;
                const int4 va = *reinterpret_cast<const int4*>(a8 + (size_t)(st * kBM + row) * kBK + col);
                const int4 vb = *reinterpret_cast<const int4*>(b8 + (size_t)(st * kBN + row) * kBK + col);
                uint4 ha0, ha1, hb0, hb1;
                i8x4_to_f16x2((uint32_t)va.x, ha0.x, ha0.y);
                i8x4_to_f16x2((uint32_t)va.y, ha0.z, ha0.w);
                i8x4_to_f16x2((uint32_t)va.z, ha1.x, ha1.y);
                i8x4_to_f16x2((uint32_t)va.w, ha1.z, ha1.w);
                i8x4_to_f16x2((uint32_t)vb.x, hb0.x, hb0.y);
                i8x4_to_f16x2((uint32_t)vb.y, hb0.z, hb0.w);
                i8x4_to_f16x2((uint32_t)vb.z, hb1.x, hb1.y);
                i8x4_to_f16x2((uint32_t)vb.w, hb1.z, hb1.w);
                *reinterpret_cast<uint4*>(ah + (size_t)row * kHP + col) = ha0;
                *reinterpret_cast<uint4*>(ah + (size_t)row * kHP + col + 8) = ha1;
                *reinterpret_cast<uint4*>(bh + (size_t)row * kHP + col) = hb0;
                *reinterpret_cast<uint4*>(bh + (size_t)row * kHP + col + 8) = hb1;
            }
        }
        __syncthreads();   // FP16 tiles complete
#pragma unroll
        for (int kq = 0; kq < kBK / 16; ++kq) {
            uint32_t af[4][4], bf[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                ldsm_x4(a_lane + (uint32_t)((i * 16 * kHP + kq * 16) * 2), af[i][0], af[i][1], af[i][2],
                        af[i][3]);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
                ldsm_x4(b_lane + (uint32_t)((jj * 16 * kHP + kq * 16) * 2), bf[2 * jj][0], bf[2 * jj][1],
                        bf[2 * jj + 1][0], bf[2 * jj + 1][1]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_f16(acc[i][j], af[i][0], af[i][1], af[i][2], af[i][3], bf[j][0], bf[j][1]);
        }
        if ((s + 1) % kChunkSteps == 0 || s + 1 == steps) {
            // exact float32 chunk -> this thread's INT32 elements of the tile
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = wm * 64 + i * 16 + g + ((e >> 1) << 3);
                        const int c = wn * 32 + j * 8 + 2 * t + (e & 1);
                        sc[r * kCP + c] += __float2int_rn(acc[i][j][e]);
                        acc[i][j][e] = 0.0f;
                    }
        }
    }
    __syncthreads();
    for (int i = tid; i < kBM * kBN / 4; i += kGemmThreads) {
        const int r = (i * 4) / kBN, c = (i * 4) % kBN;
        if (m0 + r >= M) continue;
        const int4 v = *reinterpret_cast<const int4*>(sc + r * kCP + c);
        int32_t* dst = C + (size_t)(m0 + r) * ldc + n0 + c;
        if (n0 + c + 3 < N && (ldc & 3) == 0) {
            *reinterpret_cast<int4*>(dst) = v;
        } else {
            if (n0 + c < N) dst[0] = v.x;
            if (n0 + c + 1 < N) dst[1] = v.y;
            if (n0 + c + 2 < N) dst[2] = v.z;
            if (n0 + c + 3 < N) dst[3] = v.w;
        }
    }
}

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
        const f2 e = f2_exp(f2_make(-fabsf(gv)));
        f2 num = two_prod(gv, uv);
        if (gv < 0.0f) num = f2_mul(num, e);
        p.y[(size_t)b * p.ldy + o] = f2_to_bf16(f2_div(num, f2_addf(e, 1.0f)));
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

bool gemm_supported(int K, int k_splits) { return K > 0 && K % (kBK * k_splits) == 0; }

size_t gemm_acc_bytes(int M, int N, int epilogue, int k_splits) {
    const size_t cols = (size_t)(epilogue == EPI_SWIGLU ? 2 * N : N);
    return (size_t)k_splits * M * cols * 4;
}

cudaError_t launch_gemm_projection(int epilogue, int k_splits, const GemvParams& p, int32_t* acc,
                                   const Launch& L) {
    if (p.M <= 0) return cudaSuccess;
    if (!p.xq || !p.x_scale || !gemm_supported(p.K, k_splits)) return cudaErrorInvalidValue;
    if (epilogue == EPI_SWIGLU && k_splits != 1) return cudaErrorInvalidValue;
    const int Nc = epilogue == EPI_SWIGLU ? 2 * p.N : p.N;
    const size_t smem = gemm_smem().total;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(gemm_i8_kernel), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(gemm_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    const dim3 grid((p.M + kBM - 1) / kBM, (Nc + kBN - 1) / kBN);
    const int Ks = p.K / k_splits;
    static const bool use_mma_sync = [] {
        const char* v = std::getenv("A8W8_GEMM");
        return v && v[0] == 'm';
    }();
    for (int s = 0; s < k_splits; ++s) {
        cudaError_t e = use_mma_sync
                            ? launch_pdl(gemm_i8_kernel, grid, dim3(kGemmThreads), smem, L, p.xq, p.K,
                                         p.W, p.K, p.M, Nc, s * Ks, (s + 1) * Ks,
                                         acc + (size_t)s * p.M * Nc, Nc)
                            : launch_gemm_tc(p.xq, p.M, p.W, Nc, p.K, s * Ks, (s + 1) * Ks,
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
