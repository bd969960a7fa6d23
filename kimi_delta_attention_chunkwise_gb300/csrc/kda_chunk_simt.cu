// kda_chunk_simt.cu -- fp32 CUDA-core chunk engine.
//
// Serves fp32 inputs (where bf16 tensor-core operands would be too coarse),
// head widths 16/32/64/128 and chunk sizes 16/32/64, and acts as a second,
// independent GPU witness for the tensor-core engine.
//
// Each CTA owns one (sequence, head, 32-wide value tile) chain and walks its
// chunks in order, following "Kimi Unveils Delta Attention and K3
// Architecture Updates", sec. 6:
//   6.1  G = chunk-local cumulative log decay per key channel;
//   6.3  rho_ij = beta_i sum_d k_jd k_id exp(G_id - G_jd)   (j < i),
//   6.5  chi_ij = s    sum_d k_jd q_id exp(G_id - G_jd)     (j <= i),
//        with the decay exponent taken directly per element (always <= 0,
//        so nothing overflows whatever the gates are);
//   6.2  provisional errors  e_bar_i = beta_i (v_i - S_c^T (exp(G_i) k_i));
//   6.3  causal substitution e_i = e_bar_i - sum_{j<i} rho_ij e_j;
//   6.5  o_i = s S_c^T (exp(G_i) q_i) + sum_{j<=i} chi_ij e_j;
//   6.4  S_{c+1} = Diag(exp(G_last)) S_c + sum_i (exp(G_last - G_i) k_i) e_i^T.
// The state tile stays in shared memory in fp32 for the whole sequence.
#include <cstdint>
#include <cuda_bf16.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_f32(const T *p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void st_f32(T *p, float x);
template <>
__device__ __forceinline__ void st_f32<float>(float *p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_f32<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

template <int D, int C>
struct SimtCfg {
    static constexpr int BV = D < 32 ? D : 32;  // value columns per CTA
    static constexpr int DP = D + 1;            // padded row pitch (bank spread)
    static constexpr int CP = C + 1;
    static constexpr int PARTS = kThreads / BV; // split of the substitution sums
    // shared-memory carve-up, in floats
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + C * DP;
    static constexpr int OFF_G = OFF_Q + C * DP;
    static constexpr int OFF_R = OFF_G + C * DP;
    static constexpr int OFF_A = OFF_R + C * CP;
    static constexpr int OFF_S = OFF_A + C * CP;
    static constexpr int OFF_E = OFF_S + D * BV;
    static constexpr int OFF_B = OFF_E + C * BV;
    static constexpr int OFF_GL = OFF_B + C;
    static constexpr int OFF_P = OFF_GL + D;
    static constexpr int TOTAL = OFF_P + PARTS * BV;
    static constexpr size_t BYTES = sizeof(float) * TOTAL;
};

template <typename TIn, typename TOut, int D, int C>
__global__ void __launch_bounds__(kThreads)
chunk_simt_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                  const TIn *__restrict__ v, const float *__restrict__ log_alpha,
                  const float *__restrict__ beta, float scale,
                  const float *__restrict__ initial_state, const int32_t *__restrict__ cu,
                  TOut *__restrict__ out, float *__restrict__ final_state, int32_t T,
                  int32_t H, int32_t G, int32_t pro, const float *__restrict__ gbias,
                  const float *__restrict__ galog) {
    using Cfg = SimtCfg<D, C>;
    constexpr int BV = Cfg::BV, DP = Cfg::DP, CP = Cfg::CP, PARTS = Cfg::PARTS;
    extern __shared__ float sm[];
    float *Kc = sm + Cfg::OFF_K;   // [C][DP]  k, later exp(G) k
    float *Qc = sm + Cfg::OFF_Q;   // [C][DP]  q, later s exp(G) q
    float *Gc = sm + Cfg::OFF_G;   // [C][DP]  G, later exp(G_last - G) k
    float *Rm = sm + Cfg::OFF_R;   // [C][CP]  rho (strictly lower)
    float *Aq = sm + Cfg::OFF_A;   // [C][CP]  chi (lower, diagonal included)
    float *S = sm + Cfg::OFF_S;    // [D][BV]  state tile, fp32
    float *E = sm + Cfg::OFF_E;    // [C][BV]  errors
    float *Bs = sm + Cfg::OFF_B;   // [C]      beta
    float *Gl = sm + Cfg::OFF_GL;  // [D]      G at the chunk's last token
    float *Pp = sm + Cfg::OFF_P;   // [PARTS][BV] partial sums

    const int tid = threadIdx.x;
    constexpr int NT = D / BV;
    const int vt = blockIdx.x % NT, h = blockIdx.y;
    const int seq = blockIdx.x / NT;
    int32_t t_begin = 0, t_end = T;
    if (cu) {
        t_begin = min(max(cu[seq], 0), T);
        t_end = min(max(cu[seq + 1], t_begin), T);
    }
    const size_t state_off = ((size_t)seq * H + h) * D * D + (size_t)vt * BV;
    for (int idx = tid; idx < D * BV; idx += kThreads) {
        const int d = idx / BV, j = idx % BV;
        S[idx] = initial_state ? initial_state[state_off + (size_t)d * D + j] : 0.f;
    }

    const float sens = (pro & KDA_PROLOGUE_GATE) ? __expf(galog[h]) : 0.f;
    for (int32_t c0 = t_begin; c0 < t_end; c0 += C) {
        const int L = min(C, t_end - c0);
        __syncthreads();  // previous chunk's readers of Kc/Qc/Gc/E are done
        for (int idx = tid; idx < C * D; idx += kThreads) {
            const int i = idx / D, d = idx % D;
            float kv = 0.f, qv = 0.f, gv = 0.f;
            if (i < L) {
                const size_t off = ((size_t)(c0 + i) * H + h) * D + d;
                const size_t offq = ((size_t)(c0 + i) * (H / G) + h / G) * D + d;  // group's q/k
                kv = ld_f32(k + offq);
                qv = ld_f32(q + offq);
                gv = log_alpha[off];
                if (pro & KDA_PROLOGUE_GATE) gv = pro_gate(gv, sens, gbias[(size_t)h * D + d]);
            }
            Kc[i * DP + d] = kv;
            Qc[i * DP + d] = qv;
            Gc[i * DP + d] = gv;
        }
        for (int i = tid; i < C; i += kThreads) {
            float bv = i < L ? beta[(size_t)(c0 + i) * H + h] : 0.f;
            if ((pro & KDA_PROLOGUE_BETA_LOGITS) && i < L) bv = pro_sigmoid(bv);
            Bs[i] = bv;
        }
        __syncthreads();
        // the L2 prologue: each warp normalises whole token rows of k and q
        if (pro & KDA_PROLOGUE_L2NORM_QK) {
            const int lane = tid & 31;
            for (int i = tid >> 5; i < C; i += kThreads / 32) {
                float kk = 0.f, qq = 0.f;
                for (int d = lane; d < D; d += 32) {
                    kk += Kc[i * DP + d] * Kc[i * DP + d];
                    qq += Qc[i * DP + d] * Qc[i * DP + d];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    kk += __shfl_xor_sync(0xffffffffu, kk, o);
                    qq += __shfl_xor_sync(0xffffffffu, qq, o);
                }
                const float rk = rsqrtf(kk + kL2Eps), rq = rsqrtf(qq + kL2Eps);
                for (int d = lane; d < D; d += 32) {
                    Kc[i * DP + d] *= rk;
                    Qc[i * DP + d] *= rq;
                }
            }
        }
        // 6.1: cumulative log decay along the chunk (rows past L add 0).
        for (int d = tid; d < D; d += kThreads) {
            float acc = 0.f;
            for (int i = 0; i < C; ++i) {
                acc += Gc[i * DP + d];
                Gc[i * DP + d] = acc;
            }
            Gl[d] = acc;
        }
        __syncthreads();
        // 6.3 / 6.5: causal key-key and query-key coefficients.
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int i = idx / C, j = idx % C;
            float r = 0.f, a = 0.f;
            if (j <= i && i < L) {
                for (int d = 0; d < D; ++d) {
                    const float w = __expf(Gc[i * DP + d] - Gc[j * DP + d]) * Kc[j * DP + d];
                    r += w * Kc[i * DP + d];
                    a += w * Qc[i * DP + d];
                }
            }
            Rm[i * CP + j] = (j < i) ? Bs[i] * r : 0.f;
            Aq[i * CP + j] = (j <= i) ? scale * a : 0.f;
        }
        __syncthreads();
        // Boundary-facing factors (all <= 1): exp(G) k, s exp(G) q, exp(G_last - G) k.
        for (int idx = tid; idx < C * D; idx += kThreads) {
            const int i = idx / D, d = idx % D;
            const float G = Gc[i * DP + d], kv = Kc[i * DP + d];
            const float gam = __expf(G);
            Kc[i * DP + d] = gam * kv;
            Qc[i * DP + d] = scale * gam * Qc[i * DP + d];
            Gc[i * DP + d] = __expf(Gl[d] - G) * kv;
        }
        __syncthreads();
        // 6.2: provisional errors against the decayed incoming state.
        for (int idx = tid; idx < C * BV; idx += kThreads) {
            const int i = idx / BV, j = idx % BV;
            float e = 0.f;
            if (i < L) {
                float acc = 0.f;
                for (int d = 0; d < D; ++d) acc += Kc[i * DP + d] * S[d * BV + j];
                const float vv = ld_f32(v + ((size_t)(c0 + i) * H + h) * D + (size_t)vt * BV + j);
                e = Bs[i] * (vv - acc);
            }
            E[idx] = e;
        }
        __syncthreads();
        // 6.3: forward substitution, parallel over value columns and a split
        // of each row's sum.
        {
            const int j = tid % BV, part = tid / BV;
            for (int i = 1; i < L; ++i) {
                float acc = 0.f;
                for (int m = part; m < i; m += PARTS) acc += Rm[i * CP + m] * E[m * BV + j];
                Pp[part * BV + j] = acc;
                __syncthreads();
                if (tid < BV) {
                    float s = 0.f;
                    for (int p = 0; p < PARTS; ++p) s += Pp[p * BV + tid];
                    E[i * BV + tid] -= s;
                }
                __syncthreads();
            }
        }
        // 6.5: causal outputs (read after write).
        for (int idx = tid; idx < C * BV; idx += kThreads) {
            const int i = idx / BV, j = idx % BV;
            if (i < L) {
                float acc = 0.f;
                for (int d = 0; d < D; ++d) acc += Qc[i * DP + d] * S[d * BV + j];
                for (int m = 0; m <= i; ++m) acc += Aq[i * CP + m] * E[m * BV + j];
                st_f32(out + ((size_t)(c0 + i) * H + h) * D + (size_t)vt * BV + j, acc);
            }
        }
        __syncthreads();
        // 6.4: fast-forward the state tile.
        for (int idx = tid; idx < D * BV; idx += kThreads) {
            const int d = idx / BV, j = idx % BV;
            float acc = __expf(Gl[d]) * S[idx];
            for (int i = 0; i < L; ++i) acc += Gc[i * DP + d] * E[i * BV + j];
            S[idx] = acc;
        }
    }
    __syncthreads();
    if (final_state) {
        for (int idx = tid; idx < D * BV; idx += kThreads) {
            const int d = idx / BV, j = idx % BV;
            final_state[state_off + (size_t)d * D + j] = S[idx];
        }
    }
}

template <typename TIn, typename TOut, int D, int C>
cudaError_t launch_simt_t(const ChunkArgs &a, cudaStream_t stream) {
    using Cfg = SimtCfg<D, C>;
    auto kern = chunk_simt_kernel<TIn, TOut, D, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg::BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(a.N * (D / Cfg::BV)), (unsigned)a.H);
    kern<<<grid, kThreads, Cfg::BYTES, stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k),
        static_cast<const TIn *>(a.v), a.log_alpha, a.beta, a.scale, a.initial_state,
        a.cu_seqlens, static_cast<TOut *>(a.out), a.final_state, a.T, a.H, a.G, a.pro, a.gbias,
        a.galog);
    a.clock->mark(stream);
    return cudaGetLastError();
}

template <typename TIn, typename TOut, int D>
cudaError_t launch_simt_c(const ChunkArgs &a, cudaStream_t stream) {
    switch (a.C) {
        case 16: return launch_simt_t<TIn, TOut, D, 16>(a, stream);
        case 32: return launch_simt_t<TIn, TOut, D, 32>(a, stream);
        case 64: return launch_simt_t<TIn, TOut, D, 64>(a, stream);
    }
    return cudaErrorInvalidValue;
}

template <typename TIn, typename TOut>
cudaError_t launch_simt_d(const ChunkArgs &a, cudaStream_t stream) {
    switch (a.D) {
        case 16: return launch_simt_c<TIn, TOut, 16>(a, stream);
        case 32: return launch_simt_c<TIn, TOut, 32>(a, stream);
        case 64: return launch_simt_c<TIn, TOut, 64>(a, stream);
        case 128: return launch_simt_c<TIn, TOut, 128>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t stream) {
    if (a.dtype == KDA_DTYPE_BF16) {
        if (a.out_f32) return launch_simt_d<__nv_bfloat16, float>(a, stream);
        return launch_simt_d<__nv_bfloat16, __nv_bfloat16>(a, stream);
    }
    return launch_simt_d<float, float>(a, stream);
}

}  // namespace kda
