// kda_chunk_tc.cu -- tensor-core (tcgen05 / TMEM) chunk engine for bf16
// inputs, d_k = d_v = 128, chunk C = 64.
//
// The chunkwise form of "Kimi Unveils Delta Attention and K3 Architecture
// Updates", sec. 6, in the d_k x d_v layout, written with the WY
// factorisation that the page's pipeline (sec. 6.6) names: for a chunk with
// incoming state S_c and local cumulative log decay G (sec. 6.1),
//
//   R_ij   = beta_i <k_j, exp(G_i - G_j) k_i>   (j < i)        sec. 6.3
//   A^kk   = (I + R)^-1                                          sec. 6.3
//   A^qk_ij= s <k_j, exp(G_i - G_j) q_i>        (j <= i)       sec. 6.5
//   W      = A^kk Diag(beta) (exp(G) * K),  U = A^kk Diag(beta) V
//   E      = U - W S_c                (resolved errors; sec. 6.2 + 6.3)
//   O      = (s exp(G) * Q) S_c + A^qk E                         sec. 6.5
//   S_c+1  = Diag(exp(G_last)) S_c + K_end^T E,
//            K_end_i = exp(G_last - G_i) * k_i                   sec. 6.4
//
// Three launches on the caller's stream:
//   1. chunk_table  -- cu_seqlens -> first chunk index of every sequence
//                      (chunks restart at each sequence start).
//   2. chunk_prep   -- one CTA per (chunk, head), fully parallel: G, the
//                      decayed [K;Q] K^T products on the tensor core, the
//                      triangular solve, W on the tensor core, and the
//                      boundary-facing factors.  Writes bf16 operand images
//                      (already in the 128-byte-swizzled shared-memory
//                      layout) to scratch.
//   3. chunk_scan   -- one CTA per (sequence, head, 32-wide value tile):
//                      the only serial loop, over the chunks of a sequence.
//                      The fp32 state tile lives in registers; per chunk four
//                      tcgen05 MMAs ([A^kk;0](beta V), [-W;Q_hat] S_c,
//                      K_end^T E, [0;A^qk] E) and the next chunks' operands
//                      stream in with bulk async copies (double buffered).
//
// Precision: every tensor-core product accumulates in fp32 (TMEM).  The
// decayed [K;Q] K^T product takes tf32 operands (the exp factors need fp32
// range); every other operand (A^kk, A^qk, W, Q_hat, K_end, beta V, E and
// the state S_c) is fp16, whose 11-bit significand keeps the result within
// the parity bound where bf16 operands (8 bits) do not.  The state itself
// stays fp32 in registers across the whole sequence.
//
// Overflow of the factorised decay (hard part of any tensor-core form): the
// products exp(G_i - G_j) are formed as exp(G_i - G_m) * exp(G_m - G_j) with
// the mid-chunk reference m, which is exact in fp32/bf16 range as long as
// |G_i - G_m| <= 80 for every channel and row.  A chunk that breaks this
// (decays stronger than ~exp(-80) across half a chunk) takes a CUDA-core path
// that evaluates every exp(G_i - G_j) directly, so any finite gates <= 0 work.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int D = 128;        // d_k = d_v
constexpr int C = 64;         // chunk
constexpr int BV = 64;        // value columns per scan CTA
constexpr int NT = D / BV;    // value tiles per head
constexpr int MID = 32;       // reference row of the factorised decay
constexpr float kSpanLimit = 80.f;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz

// Per-(chunk, head) scratch images (f16 operands in the swizzled layout,
// fp32 gates).
constexpr uint32_t WQ_BYTES = 2 * 16384;  // [-W ; Q_hat] : 128 rows x 128 K, 2 panels
constexpr uint32_t KE_BYTES = 16384;      // K_end^T     : 128 rows x 64 K
constexpr uint32_t AK_BYTES = 8192;       // A^kk        : 64 rows x 64 K
constexpr uint32_t AQ_BYTES = 8192;       // A^qk        : 64 rows x 64 K
constexpr uint32_t GB_BYTES = 768;        // Gamma_last [128] f32, beta [64] f32

struct Scratch {
    uint8_t *wq, *ke, *ak, *aq, *gb;
    int32_t *chunk_off;  // [N + 1]
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t max_chunks(int32_t N, int32_t T) { return (size_t)T / C + (size_t)N + 1; }

Scratch carve(void *ws, int32_t N, int32_t T, int32_t H) {
    const size_t nch = max_chunks(N, T) * (size_t)H;
    uint8_t *p = static_cast<uint8_t *>(ws);
    Scratch s;
    s.wq = p; p += align256(nch * WQ_BYTES);
    s.ke = p; p += align256(nch * KE_BYTES);
    s.ak = p; p += align256(nch * AK_BYTES);
    s.aq = p; p += align256(nch * AQ_BYTES);
    s.gb = p; p += align256(nch * GB_BYTES);
    s.chunk_off = reinterpret_cast<int32_t *>(p);
    return s;
}

__device__ __forceinline__ void seq_bounds(const int32_t *cu, int32_t s, int32_t T, int32_t &a,
                                           int32_t &b) {
    if (cu) {
        a = min(max(cu[s], 0), T);
        b = min(max(cu[s + 1], a), T);
    } else {
        a = 0;
        b = T;
    }
}

// ---------------------------------------------------------------------------
// 1. chunk table: chunk_off[s] = number of chunks before sequence s
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t *cu, int32_t N,
                                                           int32_t T, int32_t *chunk_off) {
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int32_t base = 0; base < N; base += 1024) {
        const int32_t s = base + tid;
        int32_t n = 0;
        if (s < N) {
            int32_t a, b;
            seq_bounds(cu, s, T, a, b);
            n = (b - a + C - 1) / C;
        }
        int32_t x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sum[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int32_t before = carry + (warp ? warp_sum[warp - 1] : 0) + x - n;
        if (s < N) chunk_off[s] = before;
        __syncthreads();
        if (tid == 1023) carry = before + n;
        __syncthreads();
    }
    if (tid == 0) chunk_off[N] = carry;
}

// Largest s with chunk_off[s] <= c (chunk_off is non-decreasing).
__device__ __forceinline__ int32_t find_seq(const int32_t *off, int32_t N, int32_t c) {
    int32_t lo = 0, hi = N - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (off[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// 2. per-(chunk, head) preparation
// ---------------------------------------------------------------------------
// 256 threads: thread t owns key channel d = t % 128 for the tokens of one
// half chunk (t / 128).  Shared memory, with regions reused once their
// first tenant is done:
//   a1: g tile (TMA, f32 [64][128]) -> tf32 [K_tilde ; Q_tilde], 128 rows x
//       128 K in 4 panels (64 KB) -> R, X (= A^kk) and the solve's block
//       products (fp32);
//   b1: k and q tiles (TMA, bf16 [64][128] each) -> tf32 K_hat, 64 rows x
//       128 K in 4 panels (32 KB) (slow path: G f32 [64][128]) -> A^kk f16
//       panel (8 KB) and (beta Gamma K)^T f16 panel, 128 rows x 64 K (16 KB).
constexpr int kPrepThreads = 256;
constexpr int HALF = C / 2;

struct PrepSmem {
    uint8_t a1[4 * 16384];
    uint8_t b1[4 * 8192];
    float beta[C];
    float gcarry[D];   // G at token 31 of each channel
    float gmid[D];     // G at the reference token MID
    float glast[D];    // G at the chunk's last token
    uint64_t bar_in, bar_mma;
    uint32_t tmem;
};
constexpr uint32_t kOffX = C * (C + 1) * 4;        // X after R inside a1
constexpr uint32_t kOffTb = 2 * C * (C + 1) * 4;   // block products after X
constexpr uint32_t kOffA2 = 8192;                  // (beta Gamma K)^T after A^kk inside b1
constexpr uint32_t kInBytes = 2 * C * D * 2 + C * D * 4;  // k, q bf16 + g f32 tiles
static_assert(kOffTb + 3 * 16 * 17 * 4 <= 4 * 16384, "a1 reuse");
static_assert(MID == HALF, "the reference token opens the second half");

__device__ __forceinline__ void store_row_f16_image(uint8_t *img, uint32_t row,
                                                    const float (&v)[64]) {
    // one 128-byte swizzled row of a 64-wide f16 panel, 8 chunks of 16 bytes
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint4 u;
        u.x = pack_f16x2(v[ch * 8 + 0], v[ch * 8 + 1]);
        u.y = pack_f16x2(v[ch * 8 + 2], v[ch * 8 + 3]);
        u.z = pack_f16x2(v[ch * 8 + 4], v[ch * 8 + 5]);
        u.w = pack_f16x2(v[ch * 8 + 6], v[ch * 8 + 7]);
        *reinterpret_cast<uint4 *>(img + sw128_chunk(row, ch)) = u;
    }
}

// Four 16-byte chunks (32 consecutive f16 values) of one swizzled row.
__device__ __forceinline__ void store_quarter_f16_image(uint8_t *img, uint32_t row,
                                                       uint32_t chunk0, const float (&v)[32]) {
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        uint4 u;
        u.x = pack_f16x2(v[c4 * 8 + 0], v[c4 * 8 + 1]);
        u.y = pack_f16x2(v[c4 * 8 + 2], v[c4 * 8 + 3]);
        u.z = pack_f16x2(v[c4 * 8 + 4], v[c4 * 8 + 5]);
        u.w = pack_f16x2(v[c4 * 8 + 6], v[c4 * 8 + 7]);
        *reinterpret_cast<uint4 *>(img + sw128_chunk(row, chunk0 + c4)) = u;
    }
}

struct PrepMaps {
    CUtensorMap q, k, g;  // [T, H, D] viewed as {D, H, T}, box {128, 1, 64}
};

__global__ void __launch_bounds__(kPrepThreads, 2)
chunk_prep_kernel(const __grid_constant__ PrepMaps maps, const __nv_bfloat16 *__restrict__ q,
                  const __nv_bfloat16 *__restrict__ k, const float *__restrict__ beta,
                  float scale, const int32_t *__restrict__ cu, int32_t N, int32_t T, int32_t H,
                  Scratch sc, int *status) {
    extern __shared__ uint8_t smem_raw[];
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float(*R)[C + 1] = reinterpret_cast<float(*)[C + 1]>(sm.a1);
    float(*X)[C + 1] = reinterpret_cast<float(*)[C + 1]>(sm.a1 + kOffX);
    float(*Tb)[16][17] = reinterpret_cast<float(*)[16][17]>(sm.a1 + kOffTb);
    uint8_t *b2 = sm.b1;            // A^kk, f16 panel
    uint8_t *a2 = sm.b1 + kOffA2;   // (beta Gamma K)^T, f16 panel

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t c = blockIdx.x, h = blockIdx.y;
    const int32_t total = sc.chunk_off[N];
    if (c >= total) return;
    const int32_t s = find_seq(sc.chunk_off, N, c);
    int32_t ta, tb;
    seq_bounds(cu, s, T, ta, tb);
    const int32_t t0 = ta + (c - sc.chunk_off[s]) * C;
    const int32_t L = min(C, tb - t0);
    const size_t ch = (size_t)c * H + h;
    uint8_t *wq = sc.wq + ch * WQ_BYTES;
    uint8_t *ke = sc.ke + ch * KE_BYTES;
    uint8_t *ak = sc.ak + ch * AK_BYTES;
    uint8_t *aq = sc.aq + ch * AQ_BYTES;
    float *gb = reinterpret_cast<float *>(sc.gb + ch * GB_BYTES);
    const size_t rs = (size_t)H * D;

    // Stream the chunk's k, q and log-decay tiles in (one tensor load each).
    if (tid == 0) {
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&sm.bar_in, kInBytes);
        tma_load_3d(sm.b1, &maps.k, 0, h, t0, &sm.bar_in);
        tma_load_3d(sm.b1 + C * D * 2, &maps.q, 0, h, t0, &sm.bar_in);
        tma_load_3d(sm.a1, &maps.g, 0, h, t0, &sm.bar_in);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 128);
        tmem_relinquish();
        tc_fence_before();
    }
    if (tid < C) {
        const float b = tid < L ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
        sm.beta[tid] = b;
        gb[128 + tid] = b;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    bool ok = mbar_wait_bounded(&sm.bar_in, 0, kWaitCycles);

    const int d = tid & (D - 1), hf = tid >> 7, i0 = hf * HALF;
    uint32_t kp[HALF / 2], qp[HALF / 2];
    float G[HALF];
    {
        const float *gs = reinterpret_cast<const float *>(sm.a1);
        const unsigned short *ks = reinterpret_cast<const unsigned short *>(sm.b1);
        const unsigned short *qs = ks + C * D;
#pragma unroll
        for (int jj = 0; jj < HALF / 2; ++jj) {
            const int ia = i0 + 2 * jj, ib = ia + 1;
            const uint32_t k0 = ia < L ? ks[ia * D + d] : 0u, k1 = ib < L ? ks[ib * D + d] : 0u;
            const uint32_t q0 = ia < L ? qs[ia * D + d] : 0u, q1 = ib < L ? qs[ib * D + d] : 0u;
            kp[jj] = k0 | (k1 << 16);
            qp[jj] = q0 | (q1 << 16);
        }
        float acc = 0.f;
#pragma unroll
        for (int ii = 0; ii < HALF; ++ii) {
            acc += (i0 + ii < L) ? gs[(i0 + ii) * D + d] : 0.f;
            G[ii] = acc;
        }
    }
    if (hf == 0) sm.gcarry[d] = G[HALF - 1];
    __syncthreads();  // staging consumed; carries published
    if (hf == 1) {
        const float carry = sm.gcarry[d];
#pragma unroll
        for (int ii = 0; ii < HALF; ++ii) G[ii] += carry;
        sm.gmid[d] = G[0];
        sm.glast[d] = G[HALF - 1];
    }
    __syncthreads();
    const float Gm = sm.gmid[d], Gl = sm.glast[d];
    float span = 0.f;
#pragma unroll
    for (int ii = 0; ii < HALF; ++ii) span = fmaxf(span, fabsf(G[ii] - Gm));
    const int slow = __syncthreads_or(!(span <= kSpanLimit));
    auto kval = [&](int ii) {
        return __uint_as_float((ii & 1) ? (kp[ii >> 1] & 0xFFFF0000u) : (kp[ii >> 1] << 16));
    };
    auto qval = [&](int ii) {
        return __uint_as_float((ii & 1) ? (qp[ii >> 1] & 0xFFFF0000u) : (qp[ii >> 1] << 16));
    };
    uint32_t mma_phase = 0;

    if (slow) {
        // CUDA-core path: every exp(G_i - G_j) taken directly (exponent <= 0).
        float *Gs = reinterpret_cast<float *>(sm.b1);  // [64][128]
#pragma unroll
        for (int ii = 0; ii < HALF; ++ii) Gs[(i0 + ii) * D + d] = G[ii];
        __syncthreads();
        const __nv_bfloat16 *kc = k + ((size_t)t0 * H + h) * D;
        const __nv_bfloat16 *qc = q + ((size_t)t0 * H + h) * D;
        for (int i = warp; i < C; i += kPrepThreads / 32) {
            for (int j = 0; j <= i; ++j) {
                float r = 0.f, a = 0.f;
                if (i < L) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int dd = lane + 32 * m;
                        const float w = __expf(Gs[i * D + dd] - Gs[j * D + dd]) *
                                        __bfloat162float(kc[j * rs + dd]);
                        r += w * __bfloat162float(kc[i * rs + dd]);
                        a += w * __bfloat162float(qc[i * rs + dd]);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    r += __shfl_xor_sync(0xffffffffu, r, o);
                    a += __shfl_xor_sync(0xffffffffu, a, o);
                }
                if (lane == 0) {
                    R[i][j] = (j < i) ? sm.beta[i] * r : 0.f;
                    X[i][j] = scale * a;
                }
            }
            for (int j = i + 1 + lane; j < C; j += 32) {
                R[i][j] = 0.f;
                X[i][j] = 0.f;
            }
        }
        __syncthreads();
        if (tid < C) {
            float row[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) row[j] = X[tid][j];
            store_row_f16_image(aq, tid, row);
        }
        __syncthreads();
    }

    // Boundary-facing factors and the tf32 operands, token by token.
    {
        const float e_m = __expf(Gm), e_lm = __expf(Gl - Gm);
        const uint32_t pa = (d >> 5) * 16384u, pb = (d >> 5) * 8192u;
        uint8_t *qrow = wq + (d >> 6) * 16384u;
        float kend[8];
#pragma unroll
        for (int ii = 0; ii < HALF; ++ii) {
            const int i = i0 + ii;
            const float kv = kval(ii), qv = qval(ii);
            float gam, eend;
            if (!slow) {
                const float ep = __expf(G[ii] - Gm), en = __expf(Gm - G[ii]);
                gam = ep * e_m;
                eend = e_lm * en;
                *reinterpret_cast<float *>(sm.a1 + pa + sw128_offset_f32(i, d & 31)) =
                    to_tf32(kv * ep);
                *reinterpret_cast<float *>(sm.a1 + pa + sw128_offset_f32(64 + i, d & 31)) =
                    to_tf32(qv * ep);
                *reinterpret_cast<float *>(sm.b1 + pb + sw128_offset_f32(i, d & 31)) =
                    to_tf32(kv * en);
            } else {
                gam = __expf(G[ii]);
                eend = __expf(Gl - G[ii]);
            }
            // Q_hat = s Gamma q -> rows 64..127 of the [-W ; Q_hat] image
            *reinterpret_cast<__half *>(qrow + sw128_offset(64 + i, d & 63)) =
                __float2half_rn(scale * gam * qv);
            kend[ii & 7] = eend * kv;
            if ((ii & 7) == 7) {
                uint4 u;
                u.x = pack_f16x2(kend[0], kend[1]); u.y = pack_f16x2(kend[2], kend[3]);
                u.z = pack_f16x2(kend[4], kend[5]); u.w = pack_f16x2(kend[6], kend[7]);
                *reinterpret_cast<uint4 *>(ke + sw128_chunk(d, i >> 3)) = u;
            }
        }
        if (hf == 0) gb[d] = slow ? __expf(Gl) : e_lm * e_m;
    }

    if (!slow) {
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // [K_tilde ; Q_tilde] K_hat^T on the tensor core (tf32): TMEM cols 0..63.
        if (tid == 0 && ok) {
            tc_fence_after();
            mma_panels<true>(tmem, smem_u32(sm.a1), 16384, smem_u32(sm.b1), 8192, 16,
                             idesc_tf32_f32(128, 64), false);
            mma_commit(&sm.bar_mma);
        }
        if (ok) ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, kWaitCycles);
        mma_phase ^= 1;
        tc_fence_after();
        // warp w reads TMEM lanes 32*(w%4).., columns 32*(w/4)..
        const int quad = warp & 3, chalf = warp >> 2, r = quad * 32 + lane;
        float v[32];
        if (ok) {
            tmem_ld32(tmem_addr(tmem, quad * 32, chalf * 32), v);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        __syncthreads();  // a1 is free: the MMA consumed its operands
        if (r < C) {
            const int i = r;  // key-key row
            const float b = sm.beta[i];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = chalf * 32 + jj;
                R[i][j] = (j < i && i < L) ? b * v[jj] : 0.f;
            }
        } else {
            const int i = r - C;  // query-key row
            float row[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = chalf * 32 + jj;
                row[jj] = (j <= i && i < L) ? scale * v[jj] : 0.f;
            }
            store_quarter_f16_image(aq, i, chalf * 4, row);
        }
    }
    for (int idx = tid; idx < C * (C + 1); idx += kPrepThreads) (&X[0][0])[idx] = 0.f;
    __syncthreads();

    // sec. 6.3: A^kk = (I + R)^-1, unit lower triangular, fp32, 16 x 16 blocks.
    if (tid < C) {
        const int b = tid >> 4, cc = tid & 15, o = b * 16;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc2 = 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m)
                if (m < r && m >= cc) acc2 += R[o + r][o + m] * x[m];
            x[r] = (r < cc) ? 0.f : (r == cc ? 1.f : -acc2);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) X[o + r][o + cc] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int dist = 1; dist < 4; ++dist) {
        const int nblk = 4 - dist;
        // T_IJ = sum_{K=J}^{I-1} R_IK X_KJ
        for (int e = tid; e < nblk * 256; e += kPrepThreads) {
            const int bi = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            const int I = bi + dist, J = bi;
            float acc2 = 0.f;
            for (int K = J; K < I; ++K) {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc2 += R[I * 16 + r][K * 16 + m] * X[K * 16 + m][J * 16 + cc];
            }
            Tb[bi][r][cc] = acc2;
        }
        __syncthreads();
        // X_IJ = -X_II T_IJ
        for (int e = tid; e < nblk * 256; e += kPrepThreads) {
            const int bi = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            const int I = bi + dist, J = bi;
            float acc2 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc2 += X[I * 16 + r][I * 16 + m] * Tb[bi][m][cc];
            X[I * 16 + r][J * 16 + cc] = -acc2;
        }
        __syncthreads();
    }
    if (tid < 2 * C) {
        const int row = tid >> 1, q4 = tid & 1;
        float v32[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v32[j] = X[row][q4 * 32 + j];
        store_quarter_f16_image(b2, row, q4 * 4, v32);
        store_quarter_f16_image(ak, row, q4 * 4, v32);
    }
    // (beta Gamma K)^T, row d, this thread's half of the tokens, f16
    {
        float bgk[32];
#pragma unroll
        for (int ii = 0; ii < HALF; ++ii) bgk[ii] = sm.beta[i0 + ii] * __expf(G[ii]) * kval(ii);
        store_quarter_f16_image(a2, d, hf * 4, bgk);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // W^T = (beta Gamma K)^T A^kk^T on the tensor core (f16): TMEM cols 64..127.
    if (tid == 0 && ok) {
        tc_fence_after();
        mma_panels(tmem + 64, smem_u32(a2), 0, smem_u32(b2), 0, 4, idesc_f16_f32(128, 64),
                   false);
        mma_commit(&sm.bar_mma);
    }
    if (ok) ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, kWaitCycles);
    tc_fence_after();
    if (ok) {
        const int quad = warp & 3, chalf = warp >> 2, dd = quad * 32 + lane;
        float v[32];
        tmem_ld32(tmem_addr(tmem, quad * 32, 64 + chalf * 32), v);
        // thread = key channel dd, v[jj] = W[i][dd] for i = 32*chalf + jj; store -W.
        uint8_t *pnl = wq + (dd >> 6) * 16384u;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj)
            *reinterpret_cast<__half *>(pnl + sw128_offset(chalf * 32 + jj, dd & 63)) =
                __float2half_rn(-v[jj]);
    } else if (tid == 0) {
        atomicExch(status, (int)KDA_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// 3. the inter-chunk scan with fused outputs
// ---------------------------------------------------------------------------
struct ScanStage {
    uint8_t wq[WQ_BYTES];        // [-W ; Q_hat]
    uint8_t ke[KE_BYTES];        // K_end^T
    uint8_t aa[3 * 8192];        // [A^kk | zeros | A^qk]
    float gb[GB_BYTES / 4];      // Gamma_last [128], beta [64]
    uint8_t pad[1024 - GB_BYTES % 1024];
};

struct ScanSmem {
    ScanStage st[2];
    // B operands in MN-major (value columns contiguous) 128-byte-swizzled
    // layout: one row of 64 f16 values per K index.
    uint8_t sb[D * 128];         // S_c:    K = 128 key rows
    uint8_t eb[C * 128];         // E:      K = 64 token rows
    uint8_t bv[C * 128];         // beta V: K = 64 token rows
    uint8_t ob[C * BV * 4];      // output tile staging for the TMA store (swizzled panels)
    uint64_t full[2];            // stage loaded (producer -> compute)
    uint64_t empty[2];           // stage released (compute -> producer)
    uint64_t mma_e, mma_s;       // MMA groups done: E; state increment and outputs
    uint32_t tmem;
    volatile int32_t abort_flag;
};

constexpr int kScanThreads = 160;  // warps 0-3 compute, warp 4 streams operands in
constexpr uint32_t kScanTmemCols = 128;  // D1 (BV columns) + D2 (BV columns)

__device__ __forceinline__ void compute_barrier() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// B operand (MN-major, SW128, N = 64): K walks 16 rows = 2048 bytes per step.
__device__ __forceinline__ void mma_kmajor_a_mn_b(uint32_t d_tmem, uint32_t a_base,
                                                  uint32_t a_panel, uint32_t b_base, int ksteps,
                                                  uint32_t idesc, bool accumulate_first) {
#pragma unroll
    for (int ks = 0; ks < ksteps; ++ks) {
        const uint32_t a = a_base + (ks >> 2) * a_panel + (ks & 3) * 32;
        const uint32_t b = b_base + ks * 2048;
        mma_half(d_tmem, sdesc_sw128(a), sdesc_sw128(b), idesc,
                 (ks > 0 || accumulate_first) ? 1u : 0u);
    }
}

// 32 consecutive f16 values (4 swizzled 16-byte chunks) of one MN-major row.
__device__ __forceinline__ void store_row32_f16(uint8_t *img, uint32_t row, uint32_t chunk0,
                                                const float *v) {
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
        uint4 u;
        u.x = pack_f16x2(v[c4 * 8 + 0], v[c4 * 8 + 1]);
        u.y = pack_f16x2(v[c4 * 8 + 2], v[c4 * 8 + 3]);
        u.z = pack_f16x2(v[c4 * 8 + 4], v[c4 * 8 + 5]);
        u.w = pack_f16x2(v[c4 * 8 + 6], v[c4 * 8 + 7]);
        *reinterpret_cast<uint4 *>(img + sw128_chunk(row, chunk0 + c4)) = u;
    }
}

template <typename TOut>
__global__ void __launch_bounds__(kScanThreads, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap out_map,
                  const __nv_bfloat16 *__restrict__ v, const float *__restrict__ initial_state,
                  const int32_t *__restrict__ cu, TOut *__restrict__ out,
                  float *__restrict__ final_state, int32_t N, int32_t T, int32_t H, Scratch sc,
                  int *status) {
    extern __shared__ uint8_t smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t seq = blockIdx.x / NT, vt = blockIdx.x % NT, h = blockIdx.y;
    int32_t ta, tb;
    seq_bounds(cu, seq, T, ta, tb);
    const int32_t c_begin = sc.chunk_off[seq];
    const int32_t n_chunks = (tb - ta + C - 1) / C;
    const size_t state_off = (((size_t)seq * H + h) * D + (tid & 127)) * D + (size_t)vt * BV;

    // state row of key channel tid (compute threads), BV value columns, fp32
    float S[BV];
    if (tid < 128 && initial_state) {
#pragma unroll
        for (int j = 0; j < BV; j += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(initial_state + state_off + j);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < BV; ++j) S[j] = 0.f;
    }

    bool ok = true;
    if (n_chunks > 0) {
        for (int stg = 0; stg < 2; ++stg) {  // the constant zero blocks
            uint4 *z = reinterpret_cast<uint4 *>(sm.st[stg].aa + 8192);
            for (int idx = tid; idx < 8192 / 16; idx += kScanThreads) z[idx] = make_uint4(0, 0, 0, 0);
        }
        if (tid == 0) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&sm.full[i], 1);
                mbar_init(&sm.empty[i], 128);  // every compute thread releases
            }
            mbar_init(&sm.mma_e, 1);
            mbar_init(&sm.mma_s, 1);
            sm.abort_flag = 0;
            fence_mbar_init();
        }
        if (warp == 0) {
            tmem_alloc(&sm.tmem, kScanTmemCols);
            tmem_relinquish();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = sm.tmem;
        constexpr uint32_t IDESC = idesc_f16_f32(128, BV) | (1u << 16);  // B MN-major

        if (warp == 4) {
            // ---------------- producer: stream each chunk's operands in ----------------
            for (int32_t n = 0; n < n_chunks; ++n) {
                const int stg = n & 1;
                if (n >= 2) {
                    const bool got = mbar_wait_bounded(&sm.empty[stg], ((n >> 1) - 1) & 1,
                                                       kWaitCycles);
                    if (!got || sm.abort_flag) {
                        sm.abort_flag = 1;
                        break;
                    }
                }
                const size_t ch = (size_t)(c_begin + n) * H + h;
                ScanStage &S_ = sm.st[stg];
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.full[stg],
                                          WQ_BYTES + KE_BYTES + AK_BYTES + AQ_BYTES + GB_BYTES);
                    bulk_g2s(S_.wq, sc.wq + ch * WQ_BYTES, WQ_BYTES, &sm.full[stg]);
                    bulk_g2s(S_.ke, sc.ke + ch * KE_BYTES, KE_BYTES, &sm.full[stg]);
                    bulk_g2s(S_.aa, sc.ak + ch * AK_BYTES, AK_BYTES, &sm.full[stg]);
                    bulk_g2s(S_.aa + 16384, sc.aq + ch * AQ_BYTES, AQ_BYTES, &sm.full[stg]);
                    bulk_g2s(S_.gb, sc.gb + ch * GB_BYTES, GB_BYTES, &sm.full[stg]);
                }
                __syncwarp();
            }
        } else {
            // ---------------- compute warps ----------------
            // value tile of a chunk: thread -> token row tid/2, 32 columns (64 B),
            // prefetched into registers one chunk ahead
            const int vi = tid >> 1, vh = tid & 1;
            uint4 vreg[4];
            auto load_v = [&](int32_t n) {
                const int32_t t0n = ta + n * C;
                if (n < n_chunks && vi < min(C, tb - t0n)) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        v + ((size_t)(t0n + vi) * H + h) * D + vt * BV + vh * 32);
#pragma unroll
                    for (int x = 0; x < 4; ++x) vreg[x] = __ldg(src + x);
                } else {
#pragma unroll
                    for (int x = 0; x < 4; ++x) vreg[x] = make_uint4(0, 0, 0, 0);
                }
            };
            // beta V of chunk n into the MN-major operand; then prefetch chunk n+1
            auto build_bv = [&](int32_t n) {
                const float b = sm.st[n & 1].gb[128 + vi];
                float f[32];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const uint32_t w[4] = {vreg[x].x, vreg[x].y, vreg[x].z, vreg[x].w};
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        f[x * 8 + 2 * y] = b * __uint_as_float(w[y] << 16);
                        f[x * 8 + 2 * y + 1] = b * __uint_as_float(w[y] & 0xFFFF0000u);
                    }
                }
                store_row32_f16(sm.bv, vi, vh * 4, f);
                load_v(n + 1);
            };

            // outputs of chunk n from D1 rows 64..127 (warps 2 and 3: token = tid - 64).
            // A full chunk goes out as one TMA tensor store from a staging tile; a
            // partial chunk (the end of a sequence) writes its valid rows directly,
            // so nothing past the sequence is touched.
            auto store_outputs = [&](uint32_t d1n, int32_t n) {
                const int32_t t0n = ta + n * C;
                const int32_t Ln = min(C, tb - t0n);
                const int i = tid - 64;
                float o0[32], o1[32];
                tmem_ld32x2(tmem_addr(d1n, warp * 32, 0), tmem_addr(d1n, warp * 32, 32), o0, o1);
                if (Ln == C) {
                    // staging: 128-byte column panels (1 for bf16, 2 for fp32), each
                    // [64 rows x 128 B] in the 128-byte swizzle the TMA store expects
                    if (tid == 64) bulk_wait_group_read<0>();  // staging free again
                    asm volatile("bar.sync 2, 64;" ::: "memory");
                    if constexpr (sizeof(TOut) == 2) {
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const float *src = c8 < 4 ? &o0[c8 * 8] : &o1[(c8 - 4) * 8];
                            uint4 u;
                            u.x = pack_bf16x2(src[0], src[1]);
                            u.y = pack_bf16x2(src[2], src[3]);
                            u.z = pack_bf16x2(src[4], src[5]);
                            u.w = pack_bf16x2(src[6], src[7]);
                            *reinterpret_cast<uint4 *>(sm.ob + sw128_chunk(i, c8)) = u;
                        }
                    } else {
#pragma unroll
                        for (int c16 = 0; c16 < 16; ++c16) {
                            const float *src = c16 < 8 ? &o0[c16 * 4] : &o1[(c16 - 8) * 4];
                            *reinterpret_cast<float4 *>(sm.ob + (c16 >> 3) * (C * 128) +
                                                        sw128_chunk(i, c16 & 7)) =
                                make_float4(src[0], src[1], src[2], src[3]);
                        }
                    }
                    fence_proxy_async();
                    asm volatile("bar.sync 2, 64;" ::: "memory");
                    if (tid == 64) {
                        constexpr int per_panel = 128 / (int)sizeof(TOut);
#pragma unroll
                        for (int pnl = 0; pnl < (int)sizeof(TOut) / 2; ++pnl)
                            tma_store_3d(&out_map, sm.ob + pnl * (C * 128),
                                         vt * BV + pnl * per_panel, h, t0n);
                        bulk_commit_group();
                    }
                } else if (i < Ln) {
                    TOut *dst = out + ((size_t)(t0n + i) * H + h) * D + vt * BV;
                    if constexpr (sizeof(TOut) == 2) {
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            uint4 u;
                            u.x = pack_bf16x2(o0[j], o0[j + 1]);
                            u.y = pack_bf16x2(o0[j + 2], o0[j + 3]);
                            u.z = pack_bf16x2(o0[j + 4], o0[j + 5]);
                            u.w = pack_bf16x2(o0[j + 6], o0[j + 7]);
                            *reinterpret_cast<uint4 *>(dst + j) = u;
                            u.x = pack_bf16x2(o1[j], o1[j + 1]);
                            u.y = pack_bf16x2(o1[j + 2], o1[j + 3]);
                            u.z = pack_bf16x2(o1[j + 4], o1[j + 5]);
                            u.w = pack_bf16x2(o1[j + 6], o1[j + 7]);
                            *reinterpret_cast<uint4 *>(dst + 32 + j) = u;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            *reinterpret_cast<float4 *>(dst + j) =
                                make_float4(o0[j], o0[j + 1], o0[j + 2], o0[j + 3]);
                            *reinterpret_cast<float4 *>(dst + 32 + j) =
                                make_float4(o1[j], o1[j + 1], o1[j + 2], o1[j + 3]);
                        }
                    }
                }
            };

            load_v(0);
            if (!mbar_wait_bounded(&sm.full[0], 0, kWaitCycles)) sm.abort_flag = 1;
            build_bv(0);
            const uint32_t d1 = tmem, d2 = tmem + BV;
            fence_proxy_async();
            compute_barrier();
            if (tid == 0 && !sm.abort_flag) {
                tc_fence_after();
                // D1 = [A^kk ; 0] (beta V) of chunk 0
                mma_kmajor_a_mn_b(d1, smem_u32(sm.st[0].aa), 0, smem_u32(sm.bv), 4, IDESC, false);
            }
            for (int32_t n = 0; n < n_chunks; ++n) {
                const int stg = n & 1;
                ScanStage &st = sm.st[stg];
                const uint32_t par = n & 1;

                // S_c operand (f16): thread = key row tid, 64 values
                store_row32_f16(sm.sb, tid, 0, &S[0]);
                store_row32_f16(sm.sb, tid, 4, &S[32]);
                fence_proxy_async();
                tc_fence_before();
                compute_barrier();
                if (sm.abort_flag) break;
                if (tid == 0) {
                    tc_fence_after();
                    // D1 += [-W ; Q_hat] S_c  -> rows 0..63: E = U - W S_c, rows 64..127: Q_hat S_c
                    mma_kmajor_a_mn_b(d1, smem_u32(st.wq), 16384, smem_u32(sm.sb), 8, IDESC,
                                      true);
                    mma_commit(&sm.mma_e);
                }
                if (warp < 2) {
                    if (!mbar_wait_bounded(&sm.mma_e, par, kWaitCycles)) sm.abort_flag = 1;
                    tc_fence_after();
                    float e0[32], e1[32];
                    tmem_ld32x2(tmem_addr(d1, warp * 32, 0), tmem_addr(d1, warp * 32, 32), e0, e1);
                    store_row32_f16(sm.eb, tid, 0, e0);
                    store_row32_f16(sm.eb, tid, 4, e1);
                }
                fence_proxy_async();
                tc_fence_before();
                compute_barrier();
                if (sm.abort_flag) break;
                if (tid == 0) {
                    tc_fence_after();
                    // D2 = K_end^T E (state increment); D1 += [0 ; A^qk] E (outputs)
                    mma_kmajor_a_mn_b(d2, smem_u32(st.ke), 0, smem_u32(sm.eb), 4, IDESC, false);
                    mma_kmajor_a_mn_b(d1, smem_u32(st.aa) + 8192, 0, smem_u32(sm.eb), 4, IDESC,
                                      true);
                    mma_commit(&sm.mma_s);
                }
                if (!mbar_wait_bounded(&sm.mma_s, par, kWaitCycles)) sm.abort_flag = 1;
                tc_fence_after();
                {
                    const float g = st.gb[tid];
                    // this thread's reads of chunk n's stage are done (MMAs completed)
                    mbar_arrive(&sm.empty[stg]);
                    float ds0[32], ds1[32];
                    tmem_ld32x2(tmem_addr(d2, warp * 32, 0), tmem_addr(d2, warp * 32, 32), ds0,
                                ds1);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        S[j] = fmaf(g, S[j], ds0[j]);
                        S[32 + j] = fmaf(g, S[32 + j], ds1[j]);
                    }
                }
                if (warp >= 2) store_outputs(d1, n);
                // next chunk's beta V, and its U on the tensor core ahead of time
                const bool more = n + 1 < n_chunks;
                if (more) {
                    if (!mbar_wait_bounded(&sm.full[(n + 1) & 1], ((n + 1) >> 1) & 1, kWaitCycles))
                        sm.abort_flag = 1;
                    build_bv(n + 1);
                    fence_proxy_async();
                }
                tc_fence_before();
                compute_barrier();
                if (sm.abort_flag) break;
                if (tid == 0 && more) {
                    tc_fence_after();
                    mma_kmajor_a_mn_b(d1, smem_u32(sm.st[(n + 1) & 1].aa), 0, smem_u32(sm.bv), 4,
                                      IDESC, false);
                }
            }
            if (tid == 64) bulk_wait_group_all();  // output tiles written
            if (sm.abort_flag) ok = false;
        }
        __syncthreads();
        if (sm.abort_flag) {
            ok = false;
            if (tid == 0) atomicExch(status, (int)KDA_ERR_TIMEOUT);
            // let copies already in flight land before the shared memory goes away
            if (tid == 0)
                for (int stg = 0; stg < 2; ++stg)
                    (void)mbar_wait_bounded(&sm.full[stg], 0, kWaitCycles / 8);
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kScanTmemCols);
        if (!ok) return;
    }
    if (final_state && tid < 128) {
#pragma unroll
        for (int j = 0; j < BV; j += 4)
            *reinterpret_cast<float4 *>(final_state + state_off + j) =
                make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
}

constexpr size_t kPrepSmem = sizeof(PrepSmem) + 1024;
constexpr size_t kScanSmem = sizeof(ScanSmem) + 1024;

}  // namespace

size_t chunk_tc_workspace_bytes(int32_t N, int32_t T, int32_t H) {
    const size_t nch = max_chunks(N, T) * (size_t)H;
    return align256(nch * WQ_BYTES) + align256(nch * KE_BYTES) + align256(nch * AK_BYTES) +
           align256(nch * AQ_BYTES) + align256(nch * GB_BYTES) +
           align256(((size_t)N + 1) * sizeof(int32_t));
}

// cuTensorMapEncodeTiled, fetched from the driver once (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [T, H, D] row-major tensor as a 3-D map {D, H, T}; box = one head's
// [64 tokens x 128 channels] tile.  Rows past T read as zero.
bool encode_tile_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t esize,
                     int32_t T, int32_t H) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
    const cuuint32_t box[3] = {(cuuint32_t)D, 1u, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t launch_chunk_tc(const ChunkArgs &a, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
    if (workspace_bytes < chunk_tc_workspace_bytes(a.N, a.T, a.H) || !workspace)
        return cudaErrorInvalidValue;
    const Scratch sc = carve(workspace, a.N, a.T, a.H);
    chunk_table_kernel<<<1, 1024, 0, stream>>>(a.cu_seqlens, a.N, a.T, sc.chunk_off);
    a.clock->mark(stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    if (a.T > 0) {
        PrepMaps maps;
        if (!encode_tile_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
            !encode_tile_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
            !encode_tile_map(&maps.g, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H))
            return cudaErrorInvalidValue;
        e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kPrepSmem);
        if (e != cudaSuccess) return e;
        const dim3 pgrid((unsigned)max_chunks(a.N, a.T), (unsigned)a.H);
        chunk_prep_kernel<<<pgrid, kPrepThreads, kPrepSmem, stream>>>(
            maps, static_cast<const __nv_bfloat16 *>(a.q),
            static_cast<const __nv_bfloat16 *>(a.k), a.beta, a.scale, a.cu_seqlens, a.N, a.T,
            a.H, sc, a.status);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    a.clock->mark(stream);

    const dim3 sgrid((unsigned)(a.N * NT), (unsigned)a.H);
    // output tiles [64 tokens x 64 columns] of one head; unused when T == 0
    CUtensorMap out_map;
    memset(&out_map, 0, sizeof(out_map));
    if (a.T > 0) {
        auto enc = tensor_map_encoder();
        const size_t es = a.out_f32 ? 4 : 2;
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.H, (cuuint64_t)a.T};
        const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)a.H * D * es};
        // one 128-byte column panel per box, 128-byte swizzle
        const cuuint32_t box[3] = {(cuuint32_t)(128 / es), 1u, (cuuint32_t)C};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        if (!enc ||
            enc(&out_map, a.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                3, a.out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (a.out_f32) {
        auto kern = chunk_scan_kernel<float>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
        if (e != cudaSuccess) return e;
        kern<<<sgrid, kScanThreads, kScanSmem, stream>>>(
            out_map, static_cast<const __nv_bfloat16 *>(a.v), a.initial_state, a.cu_seqlens,
            static_cast<float *>(a.out), a.final_state, a.N, a.T, a.H, sc, a.status);
    } else {
        auto kern = chunk_scan_kernel<__nv_bfloat16>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScanSmem);
        if (e != cudaSuccess) return e;
        kern<<<sgrid, kScanThreads, kScanSmem, stream>>>(
            out_map, static_cast<const __nv_bfloat16 *>(a.v), a.initial_state, a.cu_seqlens,
            static_cast<__nv_bfloat16 *>(a.out), a.final_state, a.N, a.T, a.H, sc, a.status);
    }
    a.clock->mark(stream);
    return cudaGetLastError();
}

}  // namespace kda
