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
// The state's value columns evolve independently (e_j needs only column j),
// so one CTA per (sequence, head, DC-wide column tile) keeps its tile of the
// fp32 state (and then of its gradient) in registers, thread = 4 columns x
// ROWS consecutive rows.  The gradients that sum over columns (dq, dk,
// dlog_alpha, dbeta) leave as per-tile partial sums that a second kernel
// adds up; with one tile per head they are written directly.  A forward sweep
// writes the state entering every CK-token chunk to scratch (checkpoints);
// the reverse sweep, chunk by chunk from the end, reloads the checkpoint,
// recomputes the chunk forward -- storing the state before each token and
// the chunk's p and e -- and then walks its tokens backwards.  The serial
// walk is latency-bound, so small problems are split into 16-column tiles
// for more CTAs with less work each.
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

template <int D, int DC>
struct BwdCfg {
    static constexpr int NTILE = D / DC;  // column tiles per head
    static constexpr int CG = DC / 4;     // float4 column groups of a tile
    static constexpr int THREADS = (CG * D < 256) ? CG * D : 256;
    static constexpr int RG = THREADS / CG;
    static constexpr int ROWS = D / RG;
    static constexpr int RG_PER_WARP = (CG < 32) ? 32 / CG : 1;
    static constexpr int SLOTS = RG / RG_PER_WARP;
    static_assert(RG * ROWS == D && NTILE * DC == D && DC <= 128, "row and column split");
};

// sum over the CG lanes that share this thread's rows (xor within aligned groups)
template <int CG>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int o = (CG < 32 ? CG : 32) / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sums of N values per lane over the 32 lanes of a warp, scattered: each
// butterfly round keeps the half of the values that this lane's side owns
// and adds the partner's copy of that half (N/2 shuffles instead of N), so
// after the rounds with offsets 16, 8, 4 and 2 a lane holds N/16 complete
// sums, those of indices base .. base + N/16 - 1 with base = N/16 times the
// lane's bits 1-4 read as a binary number (the values of lanes 2m and 2m+1
// after a last pairwise sum are the same).  N a multiple of 16.
template <int N>
__device__ __forceinline__ void warp_sum_scatter(float (&v)[N], int lane) {
    static_assert(N % 16 == 0, "four halvings");
#pragma unroll
    for (int round = 0; round < 4; ++round) {
        const int o = 16 >> round, n = N >> (round + 1);
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float keep = hi ? v[i + n] : v[i], give = hi ? v[i] : v[i + n];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, give, o);
        }
    }
#pragma unroll
    for (int i = 0; i < N / 16; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 1);
}
__device__ __forceinline__ int warp_sum_scatter_base(int lane, int per_lane) {
    return per_lane * (((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                       ((lane >> 1) & 1));
}

// dq, dk, dlog_alpha ([tiles][T, H, D]) and dbeta ([tiles][T, H]) are the
// per-tile sums over the tile's columns (the final gradients when NTILE = 1).
template <typename TIn, int D, int DC>
__global__ void __launch_bounds__(BwdCfg<D, DC>::THREADS, 1)
recurrent_bwd_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                     const TIn *__restrict__ v, const float *__restrict__ log_alpha,
                     const float *__restrict__ beta, float scale,
                     const float *__restrict__ initial_state, const int32_t *__restrict__ cu,
                     const TIn *__restrict__ d_out, const float *__restrict__ d_final,
                     float *__restrict__ dq, float *__restrict__ dk, float *__restrict__ dv,
                     float *__restrict__ dlog_alpha, float *__restrict__ dbeta,
                     float *__restrict__ d_initial, float *__restrict__ ckpt,
                     float *__restrict__ cstates, int32_t T, int32_t H) {
    using Cfg = BwdCfg<D, DC>;
    constexpr int CG = Cfg::CG, RG_PER_WARP = Cfg::RG_PER_WARP, SLOTS = Cfg::SLOTS;
    constexpr int ROWS = Cfg::ROWS, THREADS = Cfg::THREADS, NTILE = Cfg::NTILE;
    __shared__ __align__(16) float s_k[CK][D], s_q[CK][D], s_a[CK][D];   // per row
    __shared__ __align__(16) float s_v[CK][DC], s_do[CK][DC];           // per column of the tile
    __shared__ __align__(16) float s_p[CK][DC], s_e[CK][DC];
    __shared__ __align__(16) float s_red[SLOTS][DC];
    __shared__ __align__(16) float s_dp[DC];
    __shared__ float s_prod[DC];
    __shared__ float s_b[CK];

    const int tid = threadIdx.x, lane = tid & 31;
    const int cg = tid % CG, rg = tid / CG, row0 = rg * ROWS;
    const int32_t head_item = blockIdx.x / NTILE, ct = blockIdx.x % NTILE, col0 = ct * DC;
    const int32_t seq = head_item / H, h = head_item % H;
    const size_t tile_out = (size_t)ct * T * H;  // partial-sum tile offset, in (t, h) rows
    int32_t ta = 0, tb = T;
    if (cu) {
        ta = min(max(cu[seq], 0), T);
        tb = min(max(cu[seq + 1], ta), T);
    }
    const int32_t L = tb - ta, nch = (L + CK - 1) / CK;
    const size_t sdd = (size_t)D * D, stile = (size_t)D * DC;
    // checkpoint slot of chunk j: floor(ta / CK) + seq + j is unique across
    // sequences; each column tile keeps its own D x DC part
    auto ck_slot = [&](int32_t j) {
        return ckpt + (((size_t)(ta / CK + seq + j) * H + h) * NTILE + ct) * stile;
    };
    float *my_states = cstates + (size_t)blockIdx.x * CK * stile;
    // this thread's float4 of row r: in a full D x D state, or in a tile buffer
    auto tile = [&](float *base, int r) {
        return reinterpret_cast<float4 *>(base + (size_t)(row0 + r) * D + col0) + cg;
    };
    auto tbuf = [&](float *base, int r) {
        return reinterpret_cast<float4 *>(base + (size_t)(row0 + r) * DC) + cg;
    };

    // stage chunk j's per-token vectors (t0c .. t0c + nt)
    auto stage = [&](int32_t t0c, int nt, bool with_q_do) {
        for (int idx = tid; idx < nt * D; idx += THREADS) {
            const int i = idx / D, c = idx % D;
            const size_t o = ((size_t)(t0c + i) * H + h) * D + c;
            s_k[i][c] = ldf(k + o);
            s_a[i][c] = __expf(log_alpha[o]);
            if (with_q_do) s_q[i][c] = ldf(q + o);
        }
        for (int idx = tid; idx < nt * DC; idx += THREADS) {
            const int i = idx / DC, c = idx % DC;
            const size_t o = ((size_t)(t0c + i) * H + h) * D + col0 + c;
            s_v[i][c] = ldf(v + o);
            if (with_q_do) s_do[i][c] = d_out ? ldf(d_out + o) : 0.f;
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
        if (tid < DC) {
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
        for (int r = 0; r < ROWS; ++r) *tbuf(ck_slot(j), r) = s[r];
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
        for (int r = 0; r < ROWS; ++r) s[r] = *tbuf(ck_slot(j), r);
        __syncthreads();
        stage(t0c, nt, true);
        __syncthreads();
        // recompute the chunk forward, keeping the state before every token
        for (int i = 0; i < nt; ++i) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) *tbuf(my_states + (size_t)i * stile, r) = s[r];
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
                const float4 sp = *tbuf(my_states + (size_t)i * stile, r);  // S_prev
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
            if (tid < DC) {
                float dev = 0.f;
#pragma unroll
                for (int w = 0; w < SLOTS; ++w) dev += s_red[w][tid];
                const float bt = s_b[i];
                const size_t o = ((size_t)t * H + h) * D + col0 + tid;
                dv[o] = bt * dev;
                s_dp[tid] = -bt * dev;
                s_prod[tid] = dev * (s_v[i][tid] - s_p[i][tid]);
            }
            __syncthreads();
            if (tid < 32) {
                float acc = 0.f;
                for (int c = tid; c < DC; c += 32) acc += s_prod[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (tid == 0) dbeta[tile_out + (size_t)t * H + h] = acc;
            }
            const float4 dp4 = reinterpret_cast<const float4 *>(s_dp)[cg];
            if constexpr (CG == 32) {
                // a whole warp shares the rows: their sums over the tile's
                // columns by one scatter-reduction (dq, dk, dlog_alpha parts)
                float red[3 * ROWS];
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const int row = row0 + r;
                    const float a = s_a[i][row], kr = s_k[i][row];
                    const float4 sp = s[r];
                    float4 &d = ds[r];
                    // dSb = dS + k dp^T
                    d.x += kr * dp4.x; d.y += kr * dp4.y; d.z += kr * dp4.z; d.w += kr * dp4.w;
                    const float dkb =
                        a * (sp.x * dp4.x + sp.y * dp4.y + sp.z * dp4.z + sp.w * dp4.w);
                    red[r] = dq_r[r];
                    red[ROWS + r] = dka_r[r] + dkb;
                    red[2 * ROWS + r] = d.x * sp.x + d.y * sp.y + d.z * sp.z + d.w * sp.w;
                    d.x *= a; d.y *= a; d.z *= a; d.w *= a;  // dS_prev = Diag(a) dSb
                }
                warp_sum_scatter(red, lane);
                if ((lane & 1) == 0) {
                    constexpr int PER = 3 * ROWS / 16;
                    const int base = warp_sum_scatter_base(lane, PER);
#pragma unroll
                    for (int e = 0; e < PER; ++e) {
                        const int idx = base + e, which = idx / ROWS, row = row0 + idx % ROWS;
                        const size_t o = (tile_out + (size_t)t * H + h) * D + row;
                        const float x = red[e];
                        if (which == 0) dq[o] = scale * x;
                        else if (which == 1) dk[o] = x;
                        else dlog_alpha[o] = s_a[i][row] * x;
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const int row = row0 + r;
                    const float a = s_a[i][row], kr = s_k[i][row];
                    const float4 sp = s[r];
                    float4 &d = ds[r];
                    // dSb = dS + k dp^T
                    d.x += kr * dp4.x; d.y += kr * dp4.y; d.z += kr * dp4.z; d.w += kr * dp4.w;
                    const float dkb =
                        a * (sp.x * dp4.x + sp.y * dp4.y + sp.z * dp4.z + sp.w * dp4.w);
                    const float da = d.x * sp.x + d.y * sp.y + d.z * sp.z + d.w * sp.w;
                    const float q_sum = row_sum<CG>(dq_r[r]);
                    const float k_sum = row_sum<CG>(dka_r[r] + dkb);
                    const float a_sum = row_sum<CG>(da);
                    if (cg == 0) {
                        const size_t o = (tile_out + (size_t)t * H + h) * D + row;
                        dq[o] = scale * q_sum;
                        dk[o] = k_sum;
                        dlog_alpha[o] = a * a_sum;
                    }
                    d.x *= a; d.y *= a; d.z *= a; d.w *= a;  // dS_prev = Diag(a) dSb
                }
            }
        }
    }
    if (d_initial) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) *tile(d_initial + ((size_t)seq * H + h) * sdd, r) = ds[r];
    }
}

// dq, dk, dlog_alpha and dbeta from their per-tile partial sums.  Scalar
// accesses: the outputs need only 4-byte alignment.
__global__ void __launch_bounds__(256) bwd_tile_sum_kernel(const float *__restrict__ part,
                                                           float *__restrict__ dq,
                                                           float *__restrict__ dk,
                                                           float *__restrict__ dla,
                                                           float *__restrict__ db, size_t n_row,
                                                           size_t n_tok, int ntile) {
    // part: [3][ntile][n_row] (dq, dk, dlog_alpha), then [ntile][n_tok] (dbeta)
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    float *outs[3] = {dq, dk, dla};
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_row; i += stride) {
#pragma unroll
        for (int g = 0; g < 3; ++g) {
            const float *src = part + (size_t)g * ntile * n_row + i;
            float acc = src[0];
            for (int t = 1; t < ntile; ++t) acc += src[(size_t)t * n_row];
            outs[g][i] = acc;
        }
    }
    const float *pb = part + (size_t)3 * ntile * n_row;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_tok; i += stride) {
        float acc = pb[i];
        for (int t = 1; t < ntile; ++t) acc += pb[(size_t)t * n_tok + i];
        db[i] = acc;
    }
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

// Column tile width: 16 when the (sequence, head) pairs alone leave most SMs
// idle (fewer than two CTAs per SM), else the whole state width.
int32_t bwd_tile_cols(int32_t N, int32_t H, int32_t D) {
    const int sms = sm_count();
    if (D >= 32 && sms > 0 && (int64_t)N * H < 2 * (int64_t)sms) return 16;
    return D;
}

size_t partial_bytes(int32_t N, int32_t T, int32_t H, int32_t D) {
    const int32_t dc = bwd_tile_cols(N, H, D);
    if (dc == D) return 0;
    const size_t ntile = (size_t)(D / dc), rows = (size_t)T * H;
    return (3 * ntile * rows * D + ntile * rows) * sizeof(float);
}

template <typename TIn, int D, int DC>
cudaError_t launch_bwd_tile(const BwdArgs &a, cudaStream_t stream) {
    using Cfg = BwdCfg<D, DC>;
    const int64_t NH = (int64_t)a.N * a.H;
    float *ckpt = static_cast<float *>(a.workspace);
    float *cstates = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) +
                                               ckpt_bytes(a.N, a.T, a.H, D));
    float *part = cstates + (size_t)a.N * a.H * CK * (size_t)D * D;
    const size_t n_row = (size_t)a.T * a.H * D, n_tok = (size_t)a.T * a.H;
    const bool direct = Cfg::NTILE == 1;
    float *pq = direct ? a.dq : part;
    float *pk = direct ? a.dk : part + (size_t)Cfg::NTILE * n_row;
    float *pa = direct ? a.dlog_alpha : part + (size_t)2 * Cfg::NTILE * n_row;
    float *pb = direct ? a.dbeta : part + (size_t)3 * Cfg::NTILE * n_row;
    recurrent_bwd_kernel<TIn, D, DC><<<(unsigned)(NH * Cfg::NTILE), Cfg::THREADS, 0, stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k),
        static_cast<const TIn *>(a.v), a.log_alpha, a.beta, a.scale, a.initial_state,
        a.cu_seqlens, static_cast<const TIn *>(a.d_out), a.d_final_state, pq, pk, a.dv, pa, pb,
        a.d_initial_state, ckpt, cstates, a.T, a.H);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || direct || a.T == 0) return e;
    const int sms = sm_count();
    bwd_tile_sum_kernel<<<(unsigned)(sms > 0 ? 4 * sms : 608), 256, 0, stream>>>(
        part, a.dq, a.dk, a.dlog_alpha, a.dbeta, n_row, n_tok, Cfg::NTILE);
    return cudaGetLastError();
}

template <typename TIn, int D>
cudaError_t launch_bwd_t(const BwdArgs &a, cudaStream_t stream) {
    if ((int64_t)a.N * a.H == 0) return cudaSuccess;
    if constexpr (D >= 32) {
        if (bwd_tile_cols(a.N, a.H, D) == 16) return launch_bwd_tile<TIn, D, 16>(a, stream);
    }
    return launch_bwd_tile<TIn, D, D>(a, stream);
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
    return ckpt_bytes(N, T, H, D) + (size_t)N * H * CK * (size_t)D * D * sizeof(float) +
           partial_bytes(N, T, H, D);
}

cudaError_t launch_recurrent_bwd(const BwdArgs &a, cudaStream_t stream) {
    if (a.dtype == KDA_DTYPE_BF16) return launch_bwd_dtype<__nv_bfloat16>(a, stream);
    return launch_bwd_dtype<float>(a, stream);
}

}  // namespace kda
