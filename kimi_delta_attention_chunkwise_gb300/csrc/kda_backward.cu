// kda_backward.cu -- gradients of the KDA recurrence (training).
//
// The pages derive no gradients ("Kimi Unveils Delta Attention and K3
// Architecture Updates", sec. 6: the chunkwise form serves training).  This
// is reverse-mode differentiation of the token recurrence of sec. 4.1; per
// token, in reverse, with dS the gradient in the state after the token:
//
//   dS  += (s q) do^T          dq = s S do
//   dk   = dS e + Sb dp        de = dS^T k
//   db   = de . (v - p)        dv = b de,  dp = -b de
//   dSb  = dS + k dp^T         dlog_alpha_i = a_i sum_j dSb_ij S_prev_ij
//   dS   = Diag(a) dSb         (the gradient in the state before the token)
//
// where Sb = Diag(a) S_prev, p = Sb^T k, e = b (v - p).
//
// One CTA per (sequence, head) keeps the fp32 state (and then its gradient)
// in registers, thread = 4 columns x ROWS consecutive rows.  A forward sweep
// writes the state entering every CK-token chunk to scratch (checkpoints);
// the reverse sweep, chunk by chunk from the end, reloads the checkpoint,
// recomputes the chunk forward -- storing the state before each token and
// the chunk's p and e -- and then walks its tokens backwards.
#include <cstdint>
#include <cuda_bf16.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int CK = 8;  // tokens per checkpointed chunk (keeps the chunk buffers in 48 KB)
size_t ckpt_bytes(int32_t N, int32_t T, int32_t H, int32_t D);

template <typename T>
__device__ __forceinline__ float ldf(const T *p);
template <>
__device__ __forceinline__ float ldf<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

template <int D>
struct BwdCfg {
    static constexpr int CG = D / 4;
    static constexpr int THREADS = (CG * D < 256) ? CG * D : 256;
    static constexpr int RG = THREADS / CG;
    static constexpr int ROWS = D / RG;
    static constexpr int RG_PER_WARP = (CG < 32) ? 32 / CG : 1;
    static constexpr int SLOTS = RG / RG_PER_WARP;
    static_assert(RG * ROWS == D, "row split");
};

// sum over the CG lanes that share this thread's rows (xor within aligned groups)
template <int CG>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int o = (CG < 32 ? CG : 32) / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename TIn, int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
recurrent_bwd_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                     const TIn *__restrict__ v, const float *__restrict__ log_alpha,
                     const float *__restrict__ beta, float scale,
                     const float *__restrict__ initial_state, const int32_t *__restrict__ cu,
                     const TIn *__restrict__ d_out, const float *__restrict__ d_final,
                     float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dv,
                     float *__restrict__ dlog_alpha, float *__restrict__ dbeta,
                     float *__restrict__ d_initial, float *__restrict__ ckpt,
                     float *__restrict__ cstates, int32_t T, int32_t H) {
    using Cfg = BwdCfg<D>;
    constexpr int CG = Cfg::CG, RG_PER_WARP = Cfg::RG_PER_WARP, SLOTS = Cfg::SLOTS;
    constexpr int ROWS = Cfg::ROWS, THREADS = Cfg::THREADS;
    __shared__ __align__(16) float s_k[CK][D], s_q[CK][D], s_v[CK][D], s_a[CK][D], s_do[CK][D];
    __shared__ __align__(16) float s_p[CK][D], s_e[CK][D];
    __shared__ __align__(16) float s_red[SLOTS][D];
    __shared__ __align__(16) float s_dp[D];
    __shared__ float s_prod[D];
    __shared__ float s_b[CK];

    const int tid = threadIdx.x, lane = tid & 31;
    const int cg = tid % CG, rg = tid / CG, row0 = rg * ROWS;
    const int32_t seq = blockIdx.x / H, h = blockIdx.x % H;
    int32_t ta = 0, tb = T;
    if (cu) {
        ta = min(max(cu[seq], 0), T);
        tb = min(max(cu[seq + 1], ta), T);
    }
    const int32_t L = tb - ta, nch = (L + CK - 1) / CK;
    const size_t sdd = (size_t)D * D;
    // checkpoint slot of chunk j: floor(ta / CK) + seq + j is unique across sequences
    auto ck_slot = [&](int32_t j) { return ckpt + ((size_t)(ta / CK + seq + j) * H + h) * sdd; };
    float *my_states = cstates + (size_t)blockIdx.x * CK * sdd;
    auto tile = [&](float *base, int r) {  // this thread's float4 of row r
        return reinterpret_cast<float4 *>(base + (size_t)(row0 + r) * D) + cg;
    };

    // stage chunk j's per-token vectors (t0c .. t0c + nt)
    auto stage = [&](int32_t t0c, int nt, bool with_q_do) {
        for (int idx = tid; idx < nt * D; idx += THREADS) {
            const int i = idx / D, c = idx % D;
            const size_t o = ((size_t)(t0c + i) * H + h) * D + c;
            s_k[i][c] = ldf(k + o);
            s_v[i][c] = ldf(v + o);
            s_a[i][c] = __expf(log_alpha[o]);
            if (with_q_do) {
                s_q[i][c] = ldf(q + o);
                s_do[i][c] = d_out ? ldf(d_out + o) : 0.f;
            }
        }
        if (tid < nt) s_b[tid] = beta[(size_t)(t0c + tid) * H + h];
    };
    // one forward token on the register state: decay, p, e (to s_p / s_e[i] if asked), write
    auto forward_token = [&](float4 (&s)[ROWS], int i, bool keep) {
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float a = s_a[i][row0 + r], kr = s_k[i][row0 + r];
            s[r].x *= a; s[r].y *= a; s[r].z *= a; s[r].w *= a;
            pk.x += s[r].x * kr; pk.y += s[r].y * kr; pk.z += s[r].z * kr; pk.w += s[r].w * kr;
        }
#pragma unroll
        for (int o = CG; o < 32; o <<= 1) {
            pk.x += __shfl_xor_sync(0xffffffffu, pk.x, o); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, o);
            pk.z += __shfl_xor_sync(0xffffffffu, pk.z, o); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, o);
        }
        if ((tid % 32) < CG || CG >= 32)
            reinterpret_cast<float4 *>(s_red[rg / RG_PER_WARP])[cg] = pk;
        __syncthreads();
        if (tid < D) {
            float p = 0.f;
#pragma unroll
            for (int w = 0; w < SLOTS; ++w) p += s_red[w][tid];
            const float e = s_b[i] * (s_v[i][tid] - p);
            s_e[i][tid] = e;
            if (keep) s_p[i][tid] = p;
        }
        __syncthreads();
        const float4 e4 = reinterpret_cast<const float4 *>(s_e[i])[cg];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float kr = s_k[i][row0 + r];
            s[r].x += kr * e4.x; s[r].y += kr * e4.y; s[r].z += kr * e4.z; s[r].w += kr * e4.w;
        }
    };

    float4 s[ROWS];
    // ---- forward sweep: checkpoints
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        s[r] = initial_state ? *tile(const_cast<float *>(initial_state) + ((size_t)seq * H + h) * sdd, r)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int32_t j = 0; j < nch; ++j) {
        const int32_t t0c = ta + j * CK;
        const int nt = min(CK, tb - t0c);
#pragma unroll
        for (int r = 0; r < ROWS; ++r) *tile(ck_slot(j), r) = s[r];
        __syncthreads();  // the previous chunk's vectors are no longer read
        stage(t0c, nt, false);
        __syncthreads();
        for (int i = 0; i < nt; ++i) forward_token(s, i, false);
    }

    // ---- reverse sweep
    float4 ds[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        ds[r] = d_final ? *tile(const_cast<float *>(d_final) + ((size_t)seq * H + h) * sdd, r)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int32_t j = nch - 1; j >= 0; --j) {
        const int32_t t0c = ta + j * CK;
        const int nt = min(CK, tb - t0c);
#pragma unroll
        for (int r = 0; r < ROWS; ++r) s[r] = *tile(ck_slot(j), r);
        __syncthreads();
        stage(t0c, nt, true);
        __syncthreads();
        // recompute the chunk forward, keeping the state before every token
        for (int i = 0; i < nt; ++i) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) *tile(my_states + (size_t)i * sdd, r) = s[r];
            forward_token(s, i, true);
        }
        // and walk it backwards
        for (int i = nt - 1; i >= 0; --i) {
            const int32_t t = t0c + i;
            const float4 e4 = reinterpret_cast<const float4 *>(s_e[i])[cg];
            const float4 do4 = reinterpret_cast<const float4 *>(s_do[i])[cg];
            float4 de = make_float4(0.f, 0.f, 0.f, 0.f);
            float dq_r[ROWS], dka_r[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const float4 sp = *tile(my_states + (size_t)i * sdd, r);  // S_prev
                s[r] = sp;
                const int row = row0 + r;
                const float a = s_a[i][row], kr = s_k[i][row], qr = scale * s_q[i][row];
                // S_t = Diag(a) S_prev + k e^T
                const float4 st = make_float4(a * sp.x + kr * e4.x, a * sp.y + kr * e4.y,
                                              a * sp.z + kr * e4.z, a * sp.w + kr * e4.w);
                dq_r[r] = st.x * do4.x + st.y * do4.y + st.z * do4.z + st.w * do4.w;
                float4 &d = ds[r];
                d.x += qr * do4.x; d.y += qr * do4.y; d.z += qr * do4.z; d.w += qr * do4.w;
                dka_r[r] = d.x * e4.x + d.y * e4.y + d.z * e4.z + d.w * e4.w;
                de.x += d.x * kr; de.y += d.y * kr; de.z += d.z * kr; de.w += d.w * kr;
            }
#pragma unroll
            for (int o = CG; o < 32; o <<= 1) {
                de.x += __shfl_xor_sync(0xffffffffu, de.x, o); de.y += __shfl_xor_sync(0xffffffffu, de.y, o);
                de.z += __shfl_xor_sync(0xffffffffu, de.z, o); de.w += __shfl_xor_sync(0xffffffffu, de.w, o);
            }
            if ((tid % 32) < CG || CG >= 32)
                reinterpret_cast<float4 *>(s_red[rg / RG_PER_WARP])[cg] = de;
            __syncthreads();
            if (tid < D) {
                float dev = 0.f;
#pragma unroll
                for (int w = 0; w < SLOTS; ++w) dev += s_red[w][tid];
                const float bt = s_b[i];
                const size_t o = ((size_t)t * H + h) * D + tid;
                dv[o] = bt * dev;
                s_dp[tid] = -bt * dev;
                s_prod[tid] = dev * (s_v[i][tid] - s_p[i][tid]);
            }
            __syncthreads();
            if (tid < 32) {
                float acc = 0.f;
                for (int c = tid; c < D; c += 32) acc += s_prod[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (tid == 0) dbeta[(size_t)t * H + h] = acc;
            }
            const float4 dp4 = reinterpret_cast<const float4 *>(s_dp)[cg];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int row = row0 + r;
                const float a = s_a[i][row], kr = s_k[i][row];
                const float4 sp = s[r];
                float4 &d = ds[r];
                // dSb = dS + k dp^T
                d.x += kr * dp4.x; d.y += kr * dp4.y; d.z += kr * dp4.z; d.w += kr * dp4.w;
                const float dkb = a * (sp.x * dp4.x + sp.y * dp4.y + sp.z * dp4.z + sp.w * dp4.w);
                const float da = d.x * sp.x + d.y * sp.y + d.z * sp.z + d.w * sp.w;
                const float q_sum = row_sum<CG>(dq_r[r]);
                const float k_sum = row_sum<CG>(dka_r[r] + dkb);
                const float a_sum = row_sum<CG>(da);
                if (cg == 0) {
                    const size_t o = ((size_t)t * H + h) * D + row;
                    dq[o] = scale * q_sum;
                    dk[o] = k_sum;
                    dlog_alpha[o] = a * a_sum;
                }
                d.x *= a; d.y *= a; d.z *= a; d.w *= a;  // dS_prev = Diag(a) dSb
            }
            (void)lane;
        }
    }
    if (d_initial) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) *tile(d_initial + ((size_t)seq * H + h) * sdd, r) = ds[r];
    }
}

template <typename TIn, int D>
cudaError_t launch_bwd_t(const BwdArgs &a, cudaStream_t stream) {
    const int64_t NH = (int64_t)a.N * a.H;
    if (NH == 0) return cudaSuccess;
    float *ckpt = static_cast<float *>(a.workspace);
    float *cstates = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) +
                                               ckpt_bytes(a.N, a.T, a.H, D));
    recurrent_bwd_kernel<TIn, D><<<(unsigned)NH, BwdCfg<D>::THREADS, 0, stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k),
        static_cast<const TIn *>(a.v), a.log_alpha, a.beta, a.scale, a.initial_state,
        a.cu_seqlens, static_cast<const TIn *>(a.d_out), a.d_final_state, a.dq, a.dk, a.dv,
        a.dlog_alpha, a.dbeta, a.d_initial_state, ckpt, cstates, a.T, a.H);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_bwd_dtype(const BwdArgs &a, cudaStream_t stream) {
    switch (a.D) {
        case 16: return launch_bwd_t<TIn, 16>(a, stream);
        case 32: return launch_bwd_t<TIn, 32>(a, stream);
        case 64: return launch_bwd_t<TIn, 64>(a, stream);
        case 128: return launch_bwd_t<TIn, 128>(a, stream);
    }
    return cudaErrorInvalidValue;
}

// Scratch: the checkpoints (floor(T / CK) + N + 1 slots per head), then one
// chunk of states per (sequence, head).
size_t ckpt_bytes(int32_t N, int32_t T, int32_t H, int32_t D) {
    const size_t slots = (size_t)T / CK + (size_t)N + 1;
    return (slots * H * (size_t)D * D * sizeof(float) + 255) & ~size_t(255);
}

}  // namespace

size_t recurrent_bwd_workspace_bytes(int32_t N, int32_t T, int32_t H, int32_t D) {
    return ckpt_bytes(N, T, H, D) + (size_t)N * H * CK * (size_t)D * D * sizeof(float);
}

cudaError_t launch_recurrent_bwd(const BwdArgs &a, cudaStream_t stream) {
    if (a.dtype == KDA_DTYPE_BF16) return launch_bwd_dtype<__nv_bfloat16>(a, stream);
    return launch_bwd_dtype<float>(a, stream);
}

}  // namespace kda
