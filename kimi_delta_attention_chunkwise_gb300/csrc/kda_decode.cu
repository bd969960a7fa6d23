// kda_decode.cu -- one KDA decode step for a batch of independent sequences.
//
// The step is the recurrence of "Kimi Unveils Delta Attention and K3
// Architecture Updates", sec. 4.1 (five-line d_k x d_v form) and sec. 5
// (fused recurrent schedule): decay the rows of the state, predict S_bar^T k,
// correct, write k e^T, read S_t^T (scale q).  Using
//     S_t^T q = S_bar^T q + (k . q) e,
// both reductions (S_bar^T k and S_bar^T q) come out of ONE pass over the
// decayed state held in registers, and the write goes back in place, so every
// state byte crosses HBM exactly once in each direction.
//
// Work decomposition (d = d_k = d_v): one CTA per (sequence, head).  A thread
// owns a 4-column group of the state (one float4 per row) and ROWS rows
// strided by RG, so a warp's load of one row is fully coalesced (D = 128:
// 32 lanes x 16 B = one 512 B row).  Column sums over rows go through warp
// registers, then one shared-memory exchange across row groups.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cuda_bf16.h>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int D>
struct StepCfg {
    static constexpr int CG = D / 4;                                  // column groups
    static constexpr int THREADS = (CG * D < 256) ? CG * D : 256;
    static constexpr int RG = THREADS / CG;                           // row groups
    static constexpr int ROWS = D / RG;                               // rows per thread
    static_assert(RG * ROWS == D, "row split");
};

// PRO: the kernel applies an input prologue (compiled out when false)
template <typename TIn, typename TOut, int D, bool PRO>
__global__ void __launch_bounds__(StepCfg<D>::THREADS)
recurrent_step_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                      const TIn *__restrict__ v, const float *__restrict__ log_alpha,
                      const float *__restrict__ beta, float scale, float *state,
                      TOut *__restrict__ out, int32_t NH, int32_t H, int32_t G, int32_t pro,
                      const float *__restrict__ gbias, const float *__restrict__ galog) {
    using Cfg = StepCfg<D>;
    constexpr int CG = Cfg::CG, RG = Cfg::RG, ROWS = Cfg::ROWS, THREADS = Cfg::THREADS;
    __shared__ float s_k[D], s_q[D], s_alpha[D], s_e[D];
    __shared__ float s_red[2][RG][D];
    __shared__ float s_kq, s_rk, s_rq;

    const int64_t nh = blockIdx.x;  // (sequence, value head) pair; vectors are [N*H, D]
    if (nh >= NH) return;
    // q and k of this value head's group: [N * H / G, D]
    const int64_t qk = (nh / H) * (H / G) + (nh % H) / G;
    const int tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG;

    float4 *S = reinterpret_cast<float4 *>(state + nh * D * D);
    // Issue the state loads first: they are the bulk of the traffic.
    float4 s[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) s[r] = __ldcs(S + (size_t)(rg + r * RG) * CG + cg);

    const int hh = (int)(nh % H);
    if (!PRO) pro = 0;
    const float sens = (pro & KDA_PROLOGUE_GATE) ? __expf(galog[hh]) : 0.f;
    for (int i = tid; i < D; i += THREADS) {
        s_k[i] = to_f32(k[qk * D + i]);
        s_q[i] = to_f32(q[qk * D + i]);
        float lg = log_alpha[nh * D + i];
        if (pro & KDA_PROLOGUE_GATE) lg = pro_gate(lg, sens, gbias[(size_t)hh * D + i]);
        s_alpha[i] = __expf(lg);
    }
    __syncthreads();
    // k.q, and with the L2 prologue the two inverse norms: the row pass below
    // uses raw k and q, its sums are rescaled afterwards
    if (tid < 32) {
        float acc = 0.f, kk = 0.f, qq = 0.f;
        for (int i = tid; i < D; i += 32) {
            acc += s_k[i] * s_q[i];
            kk += s_k[i] * s_k[i];
            qq += s_q[i] * s_q[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
            kk += __shfl_xor_sync(0xffffffffu, kk, o);
            qq += __shfl_xor_sync(0xffffffffu, qq, o);
        }
        if (tid == 0) {
            const bool l2 = pro & KDA_PROLOGUE_L2NORM_QK;
            s_rk = l2 ? rsqrtf(kk + kL2Eps) : 1.f;
            s_rq = l2 ? rsqrtf(qq + kL2Eps) : 1.f;
            s_kq = acc * s_rk * s_rq;
        }
    }

    // Decay the rows, then both column reductions in one pass.
    float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int row = rg + r * RG;
        const float a = s_alpha[row], kr = s_k[row], qr = s_q[row];
        s[r].x *= a; s[r].y *= a; s[r].z *= a; s[r].w *= a;
        pk.x += s[r].x * kr; pk.y += s[r].y * kr; pk.z += s[r].z * kr; pk.w += s[r].w * kr;
        pq.x += s[r].x * qr; pq.y += s[r].y * qr; pq.z += s[r].z * qr; pq.w += s[r].w * qr;
    }
    // Lanes of a warp that share a column group hold different row groups
    // when CG < 32: fold them with shuffles first.
#pragma unroll
    for (int o = CG; o < 32; o <<= 1) {
        pk.x += __shfl_xor_sync(0xffffffffu, pk.x, o); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, o);
        pk.z += __shfl_xor_sync(0xffffffffu, pk.z, o); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, o);
        pq.x += __shfl_xor_sync(0xffffffffu, pq.x, o); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, o);
        pq.z += __shfl_xor_sync(0xffffffffu, pq.z, o); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, o);
    }
    constexpr int RG_PER_WARP = (CG < 32) ? 32 / CG : 1;
    if ((tid % 32) < CG || CG >= 32) {
        const int slot = rg / RG_PER_WARP;
        reinterpret_cast<float4 *>(s_red[0][slot])[cg] = pk;
        reinterpret_cast<float4 *>(s_red[1][slot])[cg] = pq;
    }
    __syncthreads();
    constexpr int SLOTS = RG / RG_PER_WARP;
    if (tid < D) {
        float p = 0.f, rq = 0.f;
#pragma unroll
        for (int w = 0; w < SLOTS; ++w) { p += s_red[0][w][tid]; rq += s_red[1][w][tid]; }
        const float bt = (pro & KDA_PROLOGUE_BETA_LOGITS) ? pro_sigmoid(beta[nh]) : beta[nh];
        const float e = bt * (to_f32(v[nh * D + tid]) - s_rk * p);
        s_e[tid] = s_rk * e;  // the write k_hat e^T, with k_hat = k / |k|
        out[nh * D + tid] = from_f32<TOut>(scale * (s_rq * rq + s_kq * e));
    }
    __syncthreads();

    // Write S_t = S_bar + k e^T back in place.
    const float4 e4 = reinterpret_cast<const float4 *>(s_e)[cg];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int row = rg + r * RG;
        const float kr = s_k[row];
        float4 x = s[r];
        x.x += kr * e4.x; x.y += kr * e4.y; x.z += kr * e4.z; x.w += kr * e4.w;
        __stcs(S + (size_t)row * CG + cg, x);
    }
}

template <typename TIn, typename TOut, int D>
cudaError_t launch_step_t(const StepArgs &a, cudaStream_t stream) {
    const int64_t NH = (int64_t)a.N * a.H;
    if (NH == 0) return cudaSuccess;
    auto kern = a.pro ? recurrent_step_kernel<TIn, TOut, D, true>
                      : recurrent_step_kernel<TIn, TOut, D, false>;
    kern<<<(unsigned)NH, StepCfg<D>::THREADS, 0, stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k),
        static_cast<const TIn *>(a.v), a.log_alpha, a.beta, a.scale, a.state,
        static_cast<TOut *>(a.out), (int32_t)NH, a.H, a.G, a.pro, a.gbias, a.galog);
    return cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_step_dtype(const StepArgs &a, cudaStream_t stream) {
    switch (a.D) {
        case 16: return launch_step_t<TIn, TOut, 16>(a, stream);
        case 32: return launch_step_t<TIn, TOut, 32>(a, stream);
        case 64: return launch_step_t<TIn, TOut, 64>(a, stream);
        case 128: return launch_step_t<TIn, TOut, 128>(a, stream);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Multi-token fused recurrent pass (the fused kernel "looping over multiple
// tokens" of "Linear Attention, From Scratch to Kimi 3", sec. 9, and the
// low-latency regime of "Kimi Unveils Delta Attention and K3 Architecture
// Updates", sec. 5): one CTA per (sequence, head) holds the state in
// registers across all of the sequence's tokens, so the state crosses HBM
// once in each direction however many tokens the sequence has.  Each token
// is the step above, with one block barrier: the row groups' partial column
// sums go through shared memory (double-buffered by token parity) and every
// thread finishes the sums of its own columns.  Blocks of 8 tokens' vectors
// are staged in shared memory, with k.q and the norms taken once per block.
// The state lives in a pool of slots; state_indices picks each sequence's
// slot (negative: the sequence is skipped).
// ---------------------------------------------------------------------------
// Thread layout of the multi-token pass: a thread owns a 4-column group and
// ROWS consecutive rows (its per-row coefficients load as vectors).
template <int D, int MAXT>
struct FwdCfg {
    static constexpr int CG = D / 4;
    static constexpr int THREADS = (CG * D < MAXT) ? CG * D : MAXT;
    static constexpr int RG = THREADS / CG;
    static constexpr int ROWS = D / RG;
    static constexpr int RG_PER_WARP = (CG < 32) ? 32 / CG : 1;
    static constexpr int SLOTS = RG / RG_PER_WARP;
    static constexpr int TB = 8;  // tokens staged in shared memory at a time
    static_assert(RG * ROWS == D, "row split");
};
constexpr int kFwdThreads = 256;

// ROWS consecutive floats of a shared-memory vector (16-byte aligned when ROWS % 4 == 0)
template <int ROWS>
__device__ __forceinline__ void load_rows(const float *src, float (&dst)[ROWS]) {
    if constexpr (ROWS % 4 == 0) {
#pragma unroll
        for (int i = 0; i < ROWS; i += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src + i);
            dst[i] = x.x; dst[i + 1] = x.y; dst[i + 2] = x.z; dst[i + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < ROWS; ++i) dst[i] = src[i];
    }
}

// Shared memory of the multi-token pass: the next item's state (bulk copy)
// and a block of TB tokens' vectors, fp32 (alpha = exp(log_alpha) already
// taken).
template <int D>
struct FwdSmem {
    using Cfg = FwdCfg<D, kFwdThreads>;
    float4 state[D * D / 4];
    float k[Cfg::TB][D], q[Cfg::TB][D], v[Cfg::TB][D], alpha[Cfg::TB][D];
    float red[2][2][Cfg::SLOTS][D];
    float beta[Cfg::TB];
    float kq[Cfg::TB], rk[Cfg::TB], rq[Cfg::TB];
    uint64_t bar;
    int32_t next;
};
constexpr long long kFwdWait = 2000000000LL;  // bounded wait on a state copy (SM clocks)

// Persistent: CTA b takes the (sequence, head) items b, b + grid, ... that
// have work, and while it runs one item's tokens the next item's state
// streams into shared memory (one bulk copy), so the state load of one item
// hides under the tokens of the one before.
template <typename TIn, typename TOut, int D, bool PRO>
__global__ void __launch_bounds__(FwdCfg<D, kFwdThreads>::THREADS)
recurrent_fwd_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                     const TIn *__restrict__ v, const float *__restrict__ log_alpha,
                     const float *__restrict__ beta, float scale, const int32_t *__restrict__ cu,
                     const int32_t *__restrict__ slots, int32_t num_slots, float *pool,
                     TOut *__restrict__ out, int32_t T, int32_t H, int32_t G, int32_t n_items,
                     int32_t pro, const float *__restrict__ gbias,
                     const float *__restrict__ galog, int *status) {
    using Cfg = FwdCfg<D, kFwdThreads>;
    constexpr int CG = Cfg::CG, ROWS = Cfg::ROWS, THREADS = Cfg::THREADS;
    constexpr int RG_PER_WARP = Cfg::RG_PER_WARP, SLOTS = Cfg::SLOTS, TB = Cfg::TB;
    extern __shared__ __align__(128) uint8_t fwd_smem_raw[];
    FwdSmem<D> &sm = *reinterpret_cast<FwdSmem<D> *>(fwd_smem_raw);

    const int tid = threadIdx.x;
    const int cg = tid % CG, rg = tid / CG, row0 = rg * ROWS;
    auto bounds = [&](int32_t seq, int32_t &ta, int32_t &tb) {
        ta = 0;
        tb = T;
        if (cu) {
            ta = min(max(cu[seq], 0), T);
            tb = min(max(cu[seq + 1], ta), T);
        }
    };
    // thread 0: the first item at or after `from` (in this CTA's stride) with
    // work; skipped sequences (negative slot) and empty ones leave their
    // state untouched, an out-of-range slot sets the status word
    auto find = [&](int32_t from) -> int32_t {
        for (int32_t it = from; it < n_items; it += (int32_t)gridDim.x) {
            int32_t ta, tb;
            bounds(it / H, ta, tb);
            const int32_t slot = slots ? slots[it / H] : it / H;
            if (slot < 0 || ta >= tb) continue;
            if (slot >= num_slots) {
                atomicExch(status, (int)KDA_ERR_INVALID_ARG);
                continue;
            }
            return it;
        }
        return -1;
    };
    auto state_of = [&](int32_t it) {
        const int32_t slot = slots ? slots[it / H] : it / H;
        return reinterpret_cast<float4 *>(pool + ((size_t)slot * H + it % H) * D * D);
    };
    if (tid == 0) {
        tc::mbar_init(&sm.bar, 1);
        tc::fence_mbar_init();
        const int32_t first = find((int32_t)blockIdx.x);
        sm.next = first;
        if (first >= 0) {
            tc::mbar_arrive_expect_tx(&sm.bar, D * D * 4);
            tc::bulk_g2s(sm.state, state_of(first), D * D * 4, &sm.bar);
        }
    }
    __syncthreads();
    int32_t item = sm.next;
    uint32_t phase = 0;
    if (!PRO) pro = 0;
    const bool l2 = pro & KDA_PROLOGUE_L2NORM_QK;
    while (item >= 0) {
        const int32_t seq = item / H, h = item % H;
        int32_t ta, tb;
        bounds(seq, ta, tb);
        float4 *S = state_of(item);
        const bool ok = tc::mbar_wait_bounded(&sm.bar, phase, kFwdWait);
        phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicExch(status, (int)KDA_ERR_TIMEOUT);
                (void)tc::mbar_wait_bounded(&sm.bar, phase ^ 1u, kFwdWait);
            }
            return;
        }
        float4 s[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) s[r] = sm.state[(row0 + r) * CG + cg];
        __syncthreads();  // the state buffer is free: the next item's copy goes out
        if (tid == 0) {
            const int32_t nx = find(item + (int32_t)gridDim.x);
            sm.next = nx;
            if (nx >= 0) {
                tc::mbar_arrive_expect_tx(&sm.bar, D * D * 4);
                tc::bulk_g2s(sm.state, state_of(nx), D * D * 4, &sm.bar);
            }
        }
        const float sens = (pro & KDA_PROLOGUE_GATE) ? __expf(galog[h]) : 0.f;
        int32_t n = 0;  // tokens done
        for (int32_t t0 = ta; t0 < tb; t0 += TB) {
            const int nt = min(TB, tb - t0);
            __syncthreads();  // the previous block's vectors are no longer read
            for (int idx = tid; idx < nt * D; idx += THREADS) {
                const int i = idx / D, c = idx % D;
                const size_t o = ((size_t)(t0 + i) * H + h) * D + c;
                const size_t oq = ((size_t)(t0 + i) * (H / G) + h / G) * D + c;  // the group's q/k
                sm.k[i][c] = to_f32(k[oq]);
                sm.q[i][c] = to_f32(q[oq]);
                sm.v[i][c] = to_f32(v[o]);
                float lg = log_alpha[o];
                if (pro & KDA_PROLOGUE_GATE) lg = pro_gate(lg, sens, gbias[(size_t)h * D + c]);
                sm.alpha[i][c] = __expf(lg);
            }
            if (tid < nt) {
                const float bt = beta[(size_t)(t0 + tid) * H + h];
                sm.beta[tid] = (pro & KDA_PROLOGUE_BETA_LOGITS) ? pro_sigmoid(bt) : bt;
            }
            __syncthreads();
            // per token of the block, one warp each: k.q and, with the L2
            // prologue, the inverse norms (the row pass uses raw k and q; its
            // sums are rescaled below)
            for (int i = tid / 32; i < nt; i += THREADS / 32) {
                const int lane = tid % 32;
                float acc = 0.f, kk = 0.f, qq = 0.f;
                for (int j = lane; j < D; j += 32) {
                    acc += sm.k[i][j] * sm.q[i][j];
                    kk += sm.k[i][j] * sm.k[i][j];
                    qq += sm.q[i][j] * sm.q[i][j];
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    acc += __shfl_xor_sync(0xffffffffu, acc, o);
                    kk += __shfl_xor_sync(0xffffffffu, kk, o);
                    qq += __shfl_xor_sync(0xffffffffu, qq, o);
                }
                if (lane == 0) {
                    const float rki = l2 ? rsqrtf(kk + kL2Eps) : 1.f;
                    const float rqi = l2 ? rsqrtf(qq + kL2Eps) : 1.f;
                    sm.rk[i] = rki;
                    sm.rq[i] = rqi;
                    sm.kq[i] = acc * rki * rqi;
                }
            }
            __syncthreads();
            for (int i = 0; i < nt; ++i, ++n) {
                const int b = n & 1;
                // decay the rows; both column reductions in one pass
                float ra[ROWS], rk[ROWS], rq[ROWS];
                load_rows<ROWS>(&sm.alpha[i][row0], ra);
                load_rows<ROWS>(&sm.k[i][row0], rk);
                load_rows<ROWS>(&sm.q[i][row0], rq);
                float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
                {
                    // packed pairs: the same IEEE operations, half the instructions
                    float2 k01 = make_float2(0.f, 0.f), k23 = k01, q01 = k01, q23 = k01;
#pragma unroll
                    for (int r = 0; r < ROWS; ++r) {
                        const float2 a2 = make_float2(ra[r], ra[r]), k2 = make_float2(rk[r], rk[r]),
                                     q2 = make_float2(rq[r], rq[r]);
                        const float2 s01 = f2_mul(make_float2(s[r].x, s[r].y), a2);
                        const float2 s23 = f2_mul(make_float2(s[r].z, s[r].w), a2);
                        s[r] = make_float4(s01.x, s01.y, s23.x, s23.y);
                        k01 = f2_fma(s01, k2, k01);
                        k23 = f2_fma(s23, k2, k23);
                        q01 = f2_fma(s01, q2, q01);
                        q23 = f2_fma(s23, q2, q23);
                    }
                    pk = make_float4(k01.x, k01.y, k23.x, k23.y);
                    pq = make_float4(q01.x, q01.y, q23.x, q23.y);
                }
#pragma unroll
                for (int o = CG; o < 32; o <<= 1) {
                    pk.x += __shfl_xor_sync(0xffffffffu, pk.x, o); pk.y += __shfl_xor_sync(0xffffffffu, pk.y, o);
                    pk.z += __shfl_xor_sync(0xffffffffu, pk.z, o); pk.w += __shfl_xor_sync(0xffffffffu, pk.w, o);
                    pq.x += __shfl_xor_sync(0xffffffffu, pq.x, o); pq.y += __shfl_xor_sync(0xffffffffu, pq.y, o);
                    pq.z += __shfl_xor_sync(0xffffffffu, pq.z, o); pq.w += __shfl_xor_sync(0xffffffffu, pq.w, o);
                }
                if ((tid % 32) < CG || CG >= 32) {
                    const int sl = rg / RG_PER_WARP;
                    reinterpret_cast<float4 *>(sm.red[b][0][sl])[cg] = pk;
                    reinterpret_cast<float4 *>(sm.red[b][1][sl])[cg] = pq;
                }
                __syncthreads();
                // every thread finishes the column sums of its own 4 columns
                // (the same sums in the same order in each row group), so no
                // second barrier hands e around; row group 0 writes the output
                float4 p4 = make_float4(0.f, 0.f, 0.f, 0.f), r4 = p4;
#pragma unroll
                for (int w = 0; w < SLOTS; ++w) {
                    const float4 a4 = reinterpret_cast<const float4 *>(sm.red[b][0][w])[cg];
                    const float4 c4 = reinterpret_cast<const float4 *>(sm.red[b][1][w])[cg];
                    p4.x += a4.x; p4.y += a4.y; p4.z += a4.z; p4.w += a4.w;
                    r4.x += c4.x; r4.y += c4.y; r4.z += c4.z; r4.w += c4.w;
                }
                const float4 v4 = reinterpret_cast<const float4 *>(sm.v[i])[cg];
                const float bi = sm.beta[i], rki = sm.rk[i];
                float4 e4;  // e = beta (v - S_bar^T k_hat), then the write k_hat e^T
                e4.x = bi * (v4.x - rki * p4.x);
                e4.y = bi * (v4.y - rki * p4.y);
                e4.z = bi * (v4.z - rki * p4.z);
                e4.w = bi * (v4.w - rki * p4.w);
                if (rg == 0) {
                    const float rqi = sm.rq[i], kqi = sm.kq[i];
                    const float o4[4] = {scale * (rqi * r4.x + kqi * e4.x), scale * (rqi * r4.y + kqi * e4.y),
                                         scale * (rqi * r4.z + kqi * e4.z), scale * (rqi * r4.w + kqi * e4.w)};
                    TOut *dst = out + ((size_t)(t0 + i) * H + h) * D + cg * 4;
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[j] = from_f32<TOut>(o4[j]);
                }
                e4.x *= rki; e4.y *= rki; e4.z *= rki; e4.w *= rki;
                // S_t = S_bar + k e^T
                const float2 e01 = make_float2(e4.x, e4.y), e23 = make_float2(e4.z, e4.w);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const float2 k2 = make_float2(rk[r], rk[r]);
                    const float2 s01 = f2_fma(k2, e01, make_float2(s[r].x, s[r].y));
                    const float2 s23 = f2_fma(k2, e23, make_float2(s[r].z, s[r].w));
                    s[r] = make_float4(s01.x, s01.y, s23.x, s23.y);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) __stcs(S + (size_t)(row0 + r) * CG + cg, s[r]);
        __syncthreads();  // every thread has read sm.next's update (written above)
        item = sm.next;
    }
}

template <typename TIn, typename TOut, int D>
cudaError_t launch_fwd_t(const RecurArgs &a, cudaStream_t stream) {
    const int64_t NH = (int64_t)a.N * a.H;
    if (NH == 0 || a.T == 0) return cudaSuccess;
    if (NH > INT32_MAX) return cudaErrorInvalidValue;
    auto kern = a.pro ? recurrent_fwd_kernel<TIn, TOut, D, true>
                      : recurrent_fwd_kernel<TIn, TOut, D, false>;
    constexpr int threads = FwdCfg<D, kFwdThreads>::THREADS;
    const size_t smem = sizeof(FwdSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) !=
            cudaSuccess)
        return cudaErrorInvalidValue;
    const int64_t grid = std::min<int64_t>(NH, (int64_t)std::max(1, sms * std::max(1, per_sm)));
    kern<<<(unsigned)grid, threads, smem, stream>>>(
        static_cast<const TIn *>(a.q), static_cast<const TIn *>(a.k),
        static_cast<const TIn *>(a.v), a.log_alpha, a.beta, a.scale, a.cu_seqlens,
        a.state_indices, a.num_slots, a.pool, static_cast<TOut *>(a.out), a.T, a.H, a.G,
        (int32_t)NH, a.pro, a.gbias, a.galog, a.status);
    return cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_fwd_dtype(const RecurArgs &a, cudaStream_t stream) {
    switch (a.D) {
        case 16: return launch_fwd_t<TIn, TOut, 16>(a, stream);
        case 32: return launch_fwd_t<TIn, TOut, 32>(a, stream);
        case 64: return launch_fwd_t<TIn, TOut, 64>(a, stream);
        case 128: return launch_fwd_t<TIn, TOut, 128>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_recurrent_step(const StepArgs &a, cudaStream_t stream) {
    if (a.dtype == KDA_DTYPE_BF16) {
        if (a.out_f32) return launch_step_dtype<__nv_bfloat16, float>(a, stream);
        return launch_step_dtype<__nv_bfloat16, __nv_bfloat16>(a, stream);
    }
    return launch_step_dtype<float, float>(a, stream);
}

cudaError_t launch_recurrent_fwd(const RecurArgs &a, cudaStream_t stream) {
    if (a.dtype == KDA_DTYPE_BF16) {
        if (a.out_f32) return launch_fwd_dtype<__nv_bfloat16, float>(a, stream);
        return launch_fwd_dtype<__nv_bfloat16, __nv_bfloat16>(a, stream);
    }
    return launch_fwd_dtype<float, float>(a, stream);
}

}  // namespace kda
