// kda_backward_grad.cu -- the per-chunk gradient pass of the chunkwise
// backward, on the tensor cores.
//
// The pages derive no gradients ("Kimi Unveils Delta Attention and K3
// Architecture Updates", sec. 6 and 6.6: the chunkwise form serves training);
// these are the chunk form of sec. 6 differentiated by reverse mode.  For one
// chunk of one head (tokens i, j; channels a, v; G the chunk-local cumulative
// log decay, G_l its last row; A = A^kk = (I + R)^-1 and A^qk as the forward
// engine made them; B1 = Diag(beta) V, B2 = Diag(beta)(exp(G) * K),
// K_end = exp(G_l - G) * K, Q_hat = s exp(G) * Q), with S = S_c the state
// entering the chunk and dS = dS_{c+1} the gradient of the state leaving it:
//
//   U = A B1,  W = A B2,  E = U - W S                      (forward values)
//   dE   = A^qk^T dO + K_end dS
//   dQ_hat = dO S^T,   dW = -dE S^T,   dA^qk = tril_0(dO E^T),   dK_end = E dS^T
//   dA   = dE B1^T + dW B2^T,   dB1 = A^T dE,   dB2 = A^T dW
//   dR   = tril_-1(-A^T dA A^T)
//
// and through the decayed products R_ij = beta_i <k_i, exp(G_i - G_j) k_j>,
// A^qk_ij = s <q_i, exp(G_i - G_j) k_j> to q, k and G, as
//   XR_i = sum_j dR_ij exp(G_i - G_j) k_j       XQ_i = sum_j s dA^qk_ij exp(G_i - G_j) k_j
//   YY_j = sum_i (beta_i dR_ij k_i + s dA^qk_ij q_i) exp(G_i - G_j)
// (per channel), each one tensor-core product with the forward's mid-chunk
// split exp(G_i - G_j) = exp(G_i - G_32) exp(G_32 - G_j) when every
// |G_i - G_32| <= 80, else evaluated directly on the CUDA cores.  Then
//   dq = s exp(G) dQ_hat + XQ
//   dk = exp(G_l - G) dK_end + beta exp(G) dB2 + beta XR + YY
//   dv = beta dB1,  dbeta = sum_v V dB1 + sum_a exp(G) K dB2 + sum_a K XR
//   dG = Q_hat dQ_hat - K_end dK_end + B2 dB2 + beta K XR + Q XQ - K YY,
//        plus, on the chunk's last token, sum_i K_end dK_end + exp(G_l) sum_v S dS
//   dlog_alpha = the reverse cumulative sum of dG over the chunk's tokens.
//
// Two launches over the (chunk, head) items, 256 threads each, one CTA per
// SM (shared memory), all 512 TMEM columns:
//   chunk_grad_g1 -- the products with the d x d matrices S and dS: E, dE,
//                    dQ_hat, dW, dA^qk, dK_end; stores dq, dk and dlog_alpha
//                    without the second kernel's terms, and dE, dW, dA^qk as
//                    that kernel's operand images (both orientations each).
//   chunk_grad_g2 -- the C x C products: dA, dB1, dB2, A^T dA, dR, then the
//                    decayed products' gradients; stores dv and dbeta and adds
//                    its terms to dq, dk and dlog_alpha (reductions that return
//                    nothing, one per element: the sums are deterministic).
// Inputs arrive as TMA tiles (one head's 64 tokens x 128 channels), images as
// bulk copies; operands are K-major 128-byte-swizzled shared-memory panels,
// staged by the threads from those tiles or from TMEM readouts.  Every
// product with a gradient operand is kind::tf32 (gradients need fp32 range);
// the two whose operands are both forward values (U, W and W S) are
// kind::f16 on the forward's own f16 factors, as the forward computed them.
// A 64-row operand of a 128-row MMA is read with the 8 KB that follow it
// (rows 64..127 give accumulator rows that are never read).
#include <cstdint>
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int GD = 128, GC = 64, kGThreads = 256;
constexpr uint32_t U16 = 16384;             // a 128-row tf32 panel (two 64-row ones)
constexpr uint32_t P8 = 8192;               // a 64-row panel
constexpr long long kGradWait = 2000000000LL;
constexpr float kGradSpan2 = 115.f;         // |G_i - G_32| <= 80, in base 2
constexpr uint32_t kIdF16MnB = idesc_f16_f32(128, 64) | (1u << 16);  // B MN-major

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// element ii of 32 bf16 values packed in pairs
__device__ __forceinline__ float bfv(const uint32_t (&p)[16], int ii) {
    return (ii & 1) ? bf_hi(p[ii >> 1]) : bf_lo(p[ii >> 1]);
}
__device__ __forceinline__ float f16_at(const uint8_t *panel, int row, int col) {
    return __half2float(*reinterpret_cast<const __half *>(panel + sw128_offset(row, col)));
}
// fp32 element (row, col) of a K-major panel, col < 32
__device__ __forceinline__ float &f32_at(uint8_t *panel, int row, int col) {
    return *reinterpret_cast<float *>(panel + sw128_offset_f32(row, col));
}
// 32 consecutive K values of one row of a K-major tf32 panel
__device__ __forceinline__ void row32_tf32(uint8_t *panel, int row, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4 *>(panel + sw128_chunk(row, c)) =
            make_float4(tf32_operand(v[4 * c]), tf32_operand(v[4 * c + 1]),
                        tf32_operand(v[4 * c + 2]), tf32_operand(v[4 * c + 3]));
}
// The same without the rounding (values that are tf32 operands already)
__device__ __forceinline__ void row32_raw(uint8_t *panel, int row, const float (&v)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4 *>(panel + sw128_chunk(row, c)) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}
// 64 consecutive K values (two arrays of 32) of one row of a K-major f16 panel
__device__ __forceinline__ void row64_f16(uint8_t *panel, int row, const float (&v0)[32],
                                          const float (&v1)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float *v = (c < 4 ? v0 : v1) + (c & 3) * 8;
        uint4 u;
        u.x = pack_f16x2(v[0], v[1]);
        u.y = pack_f16x2(v[2], v[3]);
        u.z = pack_f16x2(v[4], v[5]);
        u.w = pack_f16x2(v[6], v[7]);
        *reinterpret_cast<uint4 *>(panel + sw128_chunk(row, c)) = u;
    }
}
__device__ __forceinline__ void zero32(float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
}

// One thread's inputs: channel ch, tokens i0 .. i0 + 31 of the chunk, read
// from the TMA tiles ([64 tokens][128 channels]; rows past the chunk's L
// tokens read as zero): G (base 2, cumulative from the chunk's first token;
// the caller adds the first half's carry), k, v, and q or dO as bf16 pairs.
struct TokenInputs {
    float G[32];
    uint32_t kp[16], vp[16], xp[16];
};

__device__ __forceinline__ void read_tiles(const float *gt, const unsigned short *kt,
                                           const unsigned short *vt, const unsigned short *xt,
                                           int ch, int i0, int L, TokenInputs &in) {
    float acc = 0.f;
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) {
        const int i = i0 + ii;
        acc = fmaf(i < L ? gt[i * GD + ch] : 0.f, kLog2e, acc);
        in.G[ii] = acc;
    }
    auto pair = [&](const unsigned short *t, int jj) -> uint32_t {
        if (!t) return 0u;
        const int ia = i0 + 2 * jj, ib = ia + 1;
        return (ia < L ? (uint32_t)t[ia * GD + ch] : 0u) |
               ((ib < L ? (uint32_t)t[ib * GD + ch] : 0u) << 16);
    };
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
        in.kp[jj] = pair(kt, jj);
        in.vp[jj] = pair(vt, jj);
        in.xp[jj] = pair(xt, jj);
    }
}

struct GradMaps {
    CUtensorMap q, k, v, d, g;  // {128, H, T}, box {128, 1, 64}
};

// Per-item image block that G1 writes and G2 bulk-copies (tf32 operands,
// rounded), in the orientation whose rows a warp writes whole (128 bytes per
// store instruction): dE (rows i, K = v; 4 x 8 KB), dW (rows i, K = a),
// s dA^qk (rows i, K = j; 2 x 8 KB) or, for items on the direct-exponent
// path, s dA^qk as exact fp32 rows [64][64] instead (its column sums
// telescope in dlog_alpha, which magnifies any rounding of it).  G2 transposes in shared
// memory what it needs the other way round.
constexpr uint32_t IM_DE = 0, IM_DW = 32768, IM_AQ = 65536, IM_AQX = 81920;
static_assert(IM_AQX + 16384 == kGradImgBytes, "image block");

// ---------------------------------------------------------------------------
// G1: the products with S and dS
// ---------------------------------------------------------------------------
// Shared arena, in 16 KB units u0..u12 (regions reused once their readers
// are done):
//   step 0: the g tile u0-1, k tile u3, v and dO tiles u4-5 (read into
//           registers), A^kk / A^qk f16 u2, dS^T u8-11 (bulk); the q tile
//           u12 (read by the epilogue)
//   step 1: dO^T (rows v, K = i) u0-1 | A^kk, A^qk f16 u2 | A^qk^T-rows tf32
//           (rows j, K = i) u3 | K_end (rows j, K = a) u4-5 | [B1 | B2] f16
//           MN-major u6-7 | dS^T (rows v, K = a) u8-11
//   step 2: -W f16 (rows i, K = a) u2 | S_c f16 image u6-7 | S (rows a, K = v)
//           tf32 panels u0, u1, u4, u5 | [dO ; dE] (rows i, K = v) u8-11
//   step 3: dS (rows a, K = v) u0-3 | E (rows j, K = v) u4-6 | S_c image u6-7
//           (read by the dG_last term) | dO in u8-11
// TMEM columns: U / E 0..127, W 128..255, dE^T 256..319 -> [dQ_hat^T | -dW^T]
// 256..383, dA^qk^T 384..447, dK_end^T 448..511.
struct G1Smem {
    uint8_t ar[13 * U16];
    float beta[GC];
    float gcarry[GD], glast[GD], gmid[GD];
    float sterm[2][GD];   // sum over a value half of dS[a][v] S[a][v]
    float kterm[2][GD];   // sum over a token half of K_end dK_end
    float tail[GD];       // sum of the second token half's dG (for dlog_alpha)
    uint64_t bar_in, bar_ld, bar_sf, bar_dsn, bar_m[4];
    uint32_t tmem;
};
constexpr uint32_t G1_DOT = 0, G1_AQ = 2 * U16, G1_AQT = 3 * U16, G1_KE = 4 * U16,
                   G1_BB = 6 * U16, G1_DST = 8 * U16;
constexpr uint32_t G1_TG = 0, G1_TK = 3 * U16, G1_TV = 4 * U16, G1_TD = 5 * U16,
                   G1_TQ = 12 * U16;
constexpr uint32_t G1_NW = 2 * U16, G1_SF = 6 * U16, G1_ODE = 8 * U16;
constexpr uint32_t G1_DSN = 0, G1_E = 4 * U16;
__device__ __forceinline__ uint32_t g1_s_panel(int p) { return (uint32_t)(p < 2 ? p : p + 2) * U16; }
constexpr size_t kG1Smem = sizeof(G1Smem) + 1024;
static_assert(kG1Smem <= 227 * 1024, "G1 shared memory");

__global__ void __launch_bounds__(kGThreads, 1)
chunk_grad_g1_kernel(const __grid_constant__ GradMaps maps, const ChunkGradArgs a) {
    extern __shared__ uint8_t smem_raw[];
    G1Smem &sm = *reinterpret_cast<G1Smem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ar = sm.ar;
    const int tid = threadIdx.x, warp = tid >> 5, quad = warp & 3;
    const int ch = tid & 127, hf = tid >> 7, i0 = hf * 32;  // channel, token half
    const size_t item = blockIdx.x;
    const int32_t H = a.H;
    const int32_t c = (int32_t)(item / (size_t)H), h = (int32_t)(item % (size_t)H);
    const int2 tok = a.chunk_tok[c];
    const int32_t t0 = tok.x, L = tok.y;
    if (L <= 0) return;
    const bool has_do = a.d_out != nullptr;
    uint8_t *img = a.img + item * (size_t)kGradImgBytes;

    if (tid == 0) {
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_ld, 1);
        mbar_init(&sm.bar_sf, 1);
        mbar_init(&sm.bar_dsn, 1);
        for (int m = 0; m < 4; ++m) mbar_init(&sm.bar_m[m], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&sm.bar_in, (has_do ? 4u : 3u) * 16384u + 32768u);
        tma_load_3d(ar + G1_TG, &maps.g, 0, h, t0, &sm.bar_in);
        tma_load_3d(ar + G1_TK, &maps.k, 0, h, t0, &sm.bar_in);
        tma_load_3d(ar + G1_TV, &maps.v, 0, h, t0, &sm.bar_in);
        if (has_do) tma_load_3d(ar + G1_TD, &maps.d, 0, h, t0, &sm.bar_in);
        // q, read only by the epilogue (a region nothing else uses)
        tma_load_3d(ar + G1_TQ, &maps.q, 0, h, t0, &sm.bar_in);
        mbar_arrive_expect_tx(&sm.bar_ld, kBwdAuxBytes + 4 * U16);
        bulk_g2s(ar + G1_AQ, a.aux + item * kBwdAuxBytes, kBwdAuxBytes, &sm.bar_ld);
        // dS^T: four 128-row panels (K = 32 key channels each), which the
        // reverse scan writes in this layout
        const uint8_t *dt = a.ds_t + item * (4 * U16);
        for (int p = 0; p < 4; ++p) bulk_g2s(ar + G1_DST + p * U16, dt + p * U16, U16, &sm.bar_ld);
        // the later loads to L2 now
        bulk_prefetch_l2(a.sst + item * (2 * U16), 2 * U16);
        bulk_prefetch_l2(a.ds_n + item * (4 * U16), 4 * U16);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 512);
        tmem_relinquish();
    }
    if (tid < GC) sm.beta[tid] = tid < L ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    const size_t rs = (size_t)H * GD;
    const size_t base = ((size_t)t0 * H + h) * GD + ch;
    tc_fence_before();
    __syncthreads();  // barrier init, TMEM address, beta
    tc_fence_after();
    bool ok = mbar_wait_bounded(&sm.bar_in, 0, kGradWait);
    TokenInputs in;
    read_tiles(reinterpret_cast<const float *>(ar + G1_TG),
               reinterpret_cast<const unsigned short *>(ar + G1_TK),
               reinterpret_cast<const unsigned short *>(ar + G1_TV),
               has_do ? reinterpret_cast<const unsigned short *>(ar + G1_TD) : nullptr, ch, i0, L,
               in);
    if (hf == 0) sm.gcarry[ch] = in.G[31];
    __syncthreads();  // the tiles are consumed; carries published
    if (hf == 1) {
        const float cy = sm.gcarry[ch];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) in.G[ii] += cy;
        sm.glast[ch] = in.G[31];
        sm.gmid[ch] = in.G[0];
    }
    __syncthreads();
    const float Gl = sm.glast[ch];
    // the second kernel's choice of path, made the same way here: only the
    // dA^qk image that path reads is written
    bool direct;
    {
        const float Gm = sm.gmid[ch];
        float span = 0.f;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) span = fmaxf(span, fabsf(in.G[ii] - Gm));
        direct = __syncthreads_or(!(span <= kGradSpan2));
    }
    const uint32_t tmem = sm.tmem;

    // ---- step 1 operands: [B1 | B2] (f16, token rows), K_end, dO^T ----
    {
        uint8_t *b1 = ar + G1_BB + (ch >> 6) * P8;
        uint8_t *b2 = ar + G1_BB + (2 + (ch >> 6)) * P8;
        uint8_t *ke = ar + G1_KE + (ch >> 5) * P8;
        float dov[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            const float kv = bfv(in.kp, ii), b = sm.beta[i];
            *reinterpret_cast<__half *>(b1 + sw128_offset(i, ch & 63)) =
                __float2half_rn(b * bfv(in.vp, ii));
            *reinterpret_cast<__half *>(b2 + sw128_offset(i, ch & 63)) =
                __float2half_rn(b * exp2_approx(in.G[ii]) * kv);
            f32_at(ke, i, ch & 31) = tf32_operand(exp2_approx(Gl - in.G[ii]) * kv);
            dov[ii] = bfv(in.xp, ii);
        }
        row32_tf32(ar + G1_DOT + hf * U16, ch, dov);
    }
    ok = mbar_wait_bounded(&sm.bar_ld, 0, kGradWait) && ok;
    {
        // A^qk^T-rows: row j holds A^qk[i][j] over i (f16 -> fp32 is exact)
        const int j = tid & 63, ib = (tid >> 6) * 16;
        const uint8_t *aqk = ar + G1_AQ + 8192;
        uint8_t *dst = ar + G1_AQT + (ib >> 5) * P8;
#pragma unroll
        for (int e = 0; e < 16; ++e) f32_at(dst, j, (ib + e) & 31) = f16_at(aqk, ib + e, j);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        // (1) [U | W] = A^kk [B1 | B2]   (f16, B MN-major; cols 0..255)
        for (int n = 0; n < 4; ++n)
            mma_kmajor_a_mn_b(tmem + n * 64, smem_u32(ar + G1_AQ), 0,
                              smem_u32(ar + G1_BB + n * P8), 4, kIdF16MnB, false);
        mma_commit(&sm.bar_m[0]);
        // (2) dE^T = dO^T A^qk + dS^T K_end^T   (cols 256..319)
        mma_panels<true>(tmem + 256, smem_u32(ar + G1_DOT), U16, smem_u32(ar + G1_AQT), P8, 8,
                         idesc_tf32_f32(128, 64), false);
        mma_panels<true>(tmem + 256, smem_u32(ar + G1_DST), U16, smem_u32(ar + G1_KE), P8, 16,
                         idesc_tf32_f32(128, 64), true);
        mma_commit(&sm.bar_m[1]);
    }

    // ---- step 2: -W (f16 rows i) and the S_c image once (1) is done ----
    ok = ok && mbar_wait_bounded(&sm.bar_m[0], 0, kGradWait);
    if (tid == 0 && ok) {
        mbar_arrive_expect_tx(&sm.bar_sf, 2 * U16);
        bulk_g2s(ar + G1_SF, a.sst + item * (2 * U16), 2 * U16, &sm.bar_sf);
    }
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (quad < 2) {
        // lane = row i (0..63), key channels 64 hf ..
        float w0[32], w1[32];
        if (ok) {
            tmem_ld32x2(tmem_addr(tmem, quad * 32, 128 + hf * 64),
                        tmem_addr(tmem, quad * 32, 128 + hf * 64 + 32), w0, w1);
        } else {
            zero32(w0);
            zero32(w1);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            w0[j] = -w0[j];
            w1[j] = -w1[j];
        }
        row64_f16(ar + G1_NW + hf * P8, ch, w0, w1);
    }
    ok = ok && mbar_wait_bounded(&sm.bar_m[1], 0, kGradWait);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    // dE^T: lane = value channel v, tokens of this half.  Into rows 64.. of
    // [dO ; dE] (dO into rows 0..63), and out as G2's dE image once the next
    // products are issued (plain global stores ahead of the operands' proxy
    // fence would hold the fence up)
    float e[32];
    {
        if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, 256 + hf * 32), e);
        else zero32(e);
        uint8_t *ode = ar + G1_ODE + (ch >> 5) * U16;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            e[ii] = tf32_operand(e[ii]);
            f32_at(ode, 64 + i, ch & 31) = e[ii];
            f32_at(ode, i, ch & 31) = bfv(in.xp, ii);
        }
    }
    ok = ok && mbar_wait_bounded(&sm.bar_sf, 0, kGradWait);
    {
        // S_c rows a = ch, value tile hf: f16 image -> tf32 panels 2 hf, 2 hf + 1
        const uint8_t *src = ar + G1_SF + hf * U16;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(src + sw128_chunk(ch, c8));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 hv = *reinterpret_cast<const __half2 *>(&w4[e]);
                f[2 * e] = __low2float(hv);
                f[2 * e + 1] = __high2float(hv);
            }
            uint8_t *pan = ar + g1_s_panel(2 * hf + (c8 >> 2));
            const int cc = (c8 & 3) * 2;
            *reinterpret_cast<float4 *>(pan + sw128_chunk(ch, cc)) =
                make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(pan + sw128_chunk(ch, cc + 1)) =
                make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        // (3) E = U - W S_c onto U (cols 0..127; f16, B = the S_c image)
        for (int vt = 0; vt < 2; ++vt)
            mma_kmajor_a_mn_b(tmem + vt * 64, smem_u32(ar + G1_NW), P8,
                              smem_u32(ar + G1_SF + vt * U16), 8, kIdF16MnB, true);
        // (4) [dQ_hat^T | -dW^T] = S_c [dO ; dE]^T   (cols 256..383)
        mma_panels<true>(tmem + 256, smem_u32(ar + g1_s_panel(0)), U16, smem_u32(ar + G1_ODE),
                         U16, 8, idesc_tf32_f32(128, 128), false);
        mma_panels<true>(tmem + 256, smem_u32(ar + g1_s_panel(2)), U16,
                         smem_u32(ar + G1_ODE + 2 * U16), U16, 8, idesc_tf32_f32(128, 128),
                         true);
        mma_commit(&sm.bar_m[2]);
    }
    {
        uint8_t *gde = img + IM_DE + (ch >> 5) * P8;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) f32_at(gde, i0 + ii, ch & 31) = e[ii];
    }

    // ---- step 3: E (rows j) and dS (rows a) ----
    ok = ok && mbar_wait_bounded(&sm.bar_m[2], 0, kGradWait);
    if (tid == 0 && ok) {
        mbar_arrive_expect_tx(&sm.bar_dsn, 4 * U16);
        bulk_g2s(ar + G1_DSN, a.ds_n + item * (4 * U16), 4 * U16, &sm.bar_dsn);
    }
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (quad < 2) {
        float e0[32], e1[32];
        if (ok) {
            tmem_ld32x2(tmem_addr(tmem, quad * 32, hf * 64), tmem_addr(tmem, quad * 32, hf * 64 + 32),
                        e0, e1);
        } else {
            zero32(e0);
            zero32(e1);
        }
        row32_tf32(ar + G1_E + (2 * hf) * P8, ch, e0);
        row32_tf32(ar + G1_E + (2 * hf + 1) * P8, ch, e1);
    }
    ok = ok && mbar_wait_bounded(&sm.bar_dsn, 0, kGradWait);
    {
        // sum_v dS[a][v] S[a][v] over value half hf (S from the f16 image)
        const uint8_t *sf = ar + G1_SF + hf * U16;
        float acc = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(sf + sw128_chunk(ch, c8));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
            const uint8_t *pan = ar + G1_DSN + (2 * hf + (c8 >> 2)) * U16;
            const int cc = (c8 & 3) * 2;
            const float4 d0 = *reinterpret_cast<const float4 *>(pan + sw128_chunk(ch, cc));
            const float4 d1 = *reinterpret_cast<const float4 *>(pan + sw128_chunk(ch, cc + 1));
            const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 hv = *reinterpret_cast<const __half2 *>(&w4[e]);
                acc = fmaf(__low2float(hv), dd[2 * e], acc);
                acc = fmaf(__high2float(hv), dd[2 * e + 1], acc);
            }
        }
        sm.sterm[hf][ch] = acc;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        // (5) dA^qk^T = E dO^T (cols 384..447): B = rows 0..63 of [dO ; dE]
        mma_panels<true>(tmem + 384, smem_u32(ar + G1_E), P8, smem_u32(ar + G1_ODE), U16, 16,
                         idesc_tf32_f32(128, 64), false);
        // (6) dK_end^T = dS E^T (cols 448..511)
        mma_panels<true>(tmem + 448, smem_u32(ar + G1_DSN), U16, smem_u32(ar + G1_E), P8, 16,
                         idesc_tf32_f32(128, 64), false);
        mma_commit(&sm.bar_m[3]);
    }
    // q for Q_hat (its tile) while the products run
    {
        const unsigned short *qt = reinterpret_cast<const unsigned short *>(ar + G1_TQ);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int ia = i0 + 2 * jj, ib = ia + 1;
            in.xp[jj] = (ia < L ? (uint32_t)qt[ia * GD + ch] : 0u) |
                        ((ib < L ? (uint32_t)qt[ib * GD + ch] : 0u) << 16);
        }
    }
    ok = ok && mbar_wait_bounded(&sm.bar_m[3], 0, kGradWait);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();

    // ---- epilogue ----
    if (quad < 2) {
        // s dA^qk[i][j] (lane = j), masked (j <= i < L): G2's two images
        float x[32];
        if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, 384 + hf * 32), x);
        else zero32(x);
        uint8_t *gaq = img + IM_AQ + (ch >> 5) * P8;
        float *gax = reinterpret_cast<float *>(img + IM_AQX) + ch;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            x[ii] = (ch <= i && i < L) ? a.scale * x[ii] : 0.f;
        }
        if (!direct) {
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) f32_at(gaq, i0 + ii, ch & 31) = tf32_operand(x[ii]);
        } else {
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) gax[(i0 + ii) * GC] = x[ii];
        }
    }
    {
        // dW = -(-dW^T)^T: G2's dW and dW^T images
        float w[32];
        if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, 320 + hf * 32), w);
        else zero32(w);
        uint8_t *gdw = img + IM_DW + (ch >> 5) * P8;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            w[ii] = -w[ii];
            f32_at(gdw, i0 + ii, ch & 31) = tf32_operand(w[ii]);
        }
    }
    float dqh[32], dke[32];
    if (ok) {
        tmem_ld32x2(tmem_addr(tmem, quad * 32, 256 + hf * 32),
                    tmem_addr(tmem, quad * 32, 448 + hf * 32), dqh, dke);
    } else {
        zero32(dqh);
        zero32(dke);
    }
    float kt = 0.f;
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) {
        const int i = i0 + ii;
        const float gam = exp2_approx(in.G[ii]), ek = exp2_approx(Gl - in.G[ii]);
        const float qhat = a.scale * gam * bfv(in.xp, ii);
        const float kend = ek * bfv(in.kp, ii);
        kt = fmaf(kend, dke[ii], kt);
        if (i < L) {
            const size_t r = base + (size_t)i * rs;
            a.dq[r] = a.scale * gam * dqh[ii];
            a.dk[r] = ek * dke[ii];
        }
        dqh[ii] = qhat * dqh[ii] - kend * dke[ii];  // dG without the second kernel's terms
    }
    sm.kterm[hf][ch] = kt;
    __syncthreads();
    {
        // dG_last onto the chunk's last token, then the reverse cumulative sum
        const float dgl = sm.kterm[0][ch] + sm.kterm[1][ch] +
                          exp2_approx(Gl) * (sm.sterm[0][ch] + sm.sterm[1][ch]);
        float acc = 0.f;
#pragma unroll
        for (int ii = 31; ii >= 0; --ii) {
            acc += dqh[ii] + (i0 + ii == L - 1 ? dgl : 0.f);
            dqh[ii] = acc;
        }
        if (hf == 1) sm.tail[ch] = acc;
        __syncthreads();
        const float add = hf == 0 ? sm.tail[ch] : 0.f;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii)
            if (i0 + ii < L) a.dlog_alpha[base + (size_t)(i0 + ii) * rs] = dqh[ii] + add;
    }
    const bool bad = __syncthreads_or(!ok);
    if (bad && tid == 0) {
        atomicExch(a.status, (int)KDA_ERR_TIMEOUT);
        // let every copy this CTA started land before its shared memory goes
        (void)mbar_wait_bounded(&sm.bar_in, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_ld, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_sf, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_dsn, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_m[3], 0, kGradWait);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// G2: the C x C products, the decayed products' gradients, the outputs
// ---------------------------------------------------------------------------
// Shared arena (16 KB units; 13.5 of them):
//   step 0: dE (rows i, K = v) u0-1, dW (rows i, K = a) u2-3 (bulk, from
//           G1); the g tile u4-5, k and v tiles u6-7, q tile u12 (read into
//           registers); A^kk f16 at u13 (8 KB)
//   step 1: + B1 (rows j, K = v) u4-5 | B2 (rows j, K = a) u6-7 | dE^T
//           (rows v, K = i) u8-9 | dW^T (rows a, K = i) u10-11 | A^T-rows
//           (rows j, K = i) u12 (the transposed ones copied in shared memory)
//   step 2: K_hat^T (rows a, K = j) u0-1 | [Q_tilde^T | K_tilde^T] u2-5 |
//           dA^T-rows (rows m, K = i) at 96 KB | A (rows n, K = m) at 120 KB |
//           s dA^qk^T-rows (rows j, K = i) at 136 KB | s dA^qk in rows 64..127
//           of [dR ; s dA^qk] (rows i, K = j) u10-11
//   step 3: T1 (rows j, K = m) at 96 KB
//   step 4: dR into rows 0..63 of u10-11 and, as beta dR^T-rows, at u12
//   direct path: G, k, q fp32 [64][128] at u0, u2, u4; dR fp32 [64][64] at
//           u12, s dA^qk fp32 [64][64] at u10; results at 96 KB
//   epilogue: dG fp32 [64][128] at 0, dbeta partials [64][129] at 32 KB
// TMEM columns: dA 0..63, dB1^T 64..127, dB2^T 128..191, T1^T 192..255,
// -dR 256..319, [X1^T | X2^T] 320..447, Y^T 448..511 (direct path: XR, XQ,
// YY themselves in 320.., 384.., 448..).
struct G2Smem {
    uint8_t ar[13 * U16 + P8];
    float beta[GC];
    float gcarry[GD], gmid[GD];
    uint64_t bar_in, bar_ld, bar_aq, bar_m[4];
    uint32_t tmem;
};
constexpr uint32_t G2_DE = 0, G2_DW = 2 * U16, G2_B1 = 4 * U16, G2_B2 = 6 * U16,
                   G2_DET = 8 * U16, G2_DWT = 10 * U16, G2_AT = 12 * U16, G2_AF = 13 * U16;
constexpr uint32_t G2_TG = 4 * U16, G2_TK = 6 * U16, G2_TV = 7 * U16, G2_TQ = 12 * U16;
constexpr uint32_t G2_KH = 0, G2_KQ = 2 * U16, G2_DAT = 98304, G2_AN = 122880, G2_T1 = 98304,
                   G2_AQT = 139264, G2_DRQ = 10 * U16, G2_DRT = 12 * U16;
constexpr uint32_t G2_GS = 0, G2_KS = 2 * U16, G2_QS = 4 * U16, G2_XS = 98304;
constexpr uint32_t G2_DGS = 0, G2_PS = 2 * U16;
constexpr int kPS = 129;  // row stride of the dbeta partials (conflict-free column sums)
constexpr size_t kG2Smem = sizeof(G2Smem) + 1024;
static_assert(kG2Smem <= 227 * 1024, "G2 shared memory");
static_assert(G2_AN + 16384 <= G2_AQT && G2_AQT + 16384 <= G2_DRQ, "step 2 regions");
static_assert(G2_XS + 2 * GC * GD * 4 <= G2_DRQ, "direct-path results below [dR ; dA^qk]");

__global__ void __launch_bounds__(kGThreads, 1)
chunk_grad_g2_kernel(const __grid_constant__ GradMaps maps, const ChunkGradArgs a) {
    extern __shared__ uint8_t smem_raw[];
    G2Smem &sm = *reinterpret_cast<G2Smem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ar = sm.ar;
    const int tid = threadIdx.x, warp = tid >> 5, quad = warp & 3;
    const int ch = tid & 127, hf = tid >> 7, i0 = hf * 32;
    const size_t item = blockIdx.x;
    const int32_t H = a.H;
    const int32_t c = (int32_t)(item / (size_t)H), h = (int32_t)(item % (size_t)H);
    const int2 tok = a.chunk_tok[c];
    const int32_t t0 = tok.x, L = tok.y;
    if (L <= 0) return;
    const uint8_t *img = a.img + item * (size_t)kGradImgBytes;

    if (tid == 0) {
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_ld, 1);
        mbar_init(&sm.bar_aq, 1);
        for (int m = 0; m < 4; ++m) mbar_init(&sm.bar_m[m], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&sm.bar_in, 3 * 16384 + 32768);
        tma_load_3d(ar + G2_TG, &maps.g, 0, h, t0, &sm.bar_in);
        tma_load_3d(ar + G2_TK, &maps.k, 0, h, t0, &sm.bar_in);
        tma_load_3d(ar + G2_TV, &maps.v, 0, h, t0, &sm.bar_in);
        tma_load_3d(ar + G2_TQ, &maps.q, 0, h, t0, &sm.bar_in);
        mbar_arrive_expect_tx(&sm.bar_ld, 2 * 32768 + 8192);
        bulk_g2s(ar + G2_DE, img + IM_DE, 32768, &sm.bar_ld);
        bulk_g2s(ar + G2_DW, img + IM_DW, 32768, &sm.bar_ld);
        bulk_g2s(ar + G2_AF, a.aux + item * kBwdAuxBytes, 8192, &sm.bar_ld);
        bulk_prefetch_l2(img + IM_AQ, 32768);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 512);
        tmem_relinquish();
    }
    if (tid < GC) sm.beta[tid] = tid < L ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    const size_t rs = (size_t)H * GD;
    const size_t base = ((size_t)t0 * H + h) * GD + ch;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = mbar_wait_bounded(&sm.bar_in, 0, kGradWait);
    TokenInputs in;
    read_tiles(reinterpret_cast<const float *>(ar + G2_TG),
               reinterpret_cast<const unsigned short *>(ar + G2_TK),
               reinterpret_cast<const unsigned short *>(ar + G2_TV),
               reinterpret_cast<const unsigned short *>(ar + G2_TQ), ch, i0, L, in);
    if (hf == 0) sm.gcarry[ch] = in.G[31];
    __syncthreads();  // tiles consumed; carries published
    if (hf == 1) {
        const float cy = sm.gcarry[ch];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) in.G[ii] += cy;
        sm.gmid[ch] = in.G[0];
    }
    __syncthreads();
    const float Gm = sm.gmid[ch];
    float span = 0.f;
#pragma unroll
    for (int ii = 0; ii < 32; ++ii) span = fmaxf(span, fabsf(in.G[ii] - Gm));
    const bool direct = __syncthreads_or(!(span <= kGradSpan2));
    // direct exponents factorised about each 16-token block's first token
    // when every block spans at most 115 (base 2: no factor leaves fp32)
    const bool blocks =
        direct && !__syncthreads_or(!(in.G[0] - in.G[15] <= kGradSpan2 &&
                                      in.G[16] - in.G[31] <= kGradSpan2));
    const uint32_t tmem = sm.tmem;

    // ---- step 1 operands: B1, B2 (token rows), A^T-rows ----
    {
        uint8_t *b1 = ar + G2_B1 + (ch >> 5) * P8, *b2 = ar + G2_B2 + (ch >> 5) * P8;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            const float b = sm.beta[i];
            f32_at(b1, i, ch & 31) = tf32_operand(b * bfv(in.vp, ii));
            f32_at(b2, i, ch & 31) = tf32_operand(b * exp2_approx(in.G[ii]) * bfv(in.kp, ii));
        }
    }
    ok = mbar_wait_bounded(&sm.bar_ld, 0, kGradWait) && ok;
    {
        // dE^T and dW^T (rows v / a, K = i) from dE and dW (rows i)
        float xe[32], xw[32];
        uint8_t *de = ar + G2_DE + (ch >> 5) * P8, *dw = ar + G2_DW + (ch >> 5) * P8;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            xe[ii] = f32_at(de, i0 + ii, ch & 31);
            xw[ii] = f32_at(dw, i0 + ii, ch & 31);
        }
        row32_raw(ar + G2_DET + hf * U16, ch, xe);
        row32_raw(ar + G2_DWT + hf * U16, ch, xw);
    }
    {
        // A^T-rows: row j holds A[i][j] over i
        const int j = tid & 63, ib = (tid >> 6) * 16;
        const uint8_t *af = ar + G2_AF;
        uint8_t *dst = ar + G2_AT + (ib >> 5) * P8;
#pragma unroll
        for (int e = 0; e < 16; ++e) f32_at(dst, j, (ib + e) & 31) = f16_at(af, ib + e, j);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        // (1) dA = dE B1^T + dW B2^T   (cols 0..63)
        mma_panels<true>(tmem, smem_u32(ar + G2_DE), P8, smem_u32(ar + G2_B1), P8, 16,
                         idesc_tf32_f32(128, 64), false);
        mma_panels<true>(tmem, smem_u32(ar + G2_DW), P8, smem_u32(ar + G2_B2), P8, 16,
                         idesc_tf32_f32(128, 64), true);
        // (2) dB1^T = dE^T A, dB2^T = dW^T A   (cols 64..127, 128..191)
        mma_panels<true>(tmem + 64, smem_u32(ar + G2_DET), U16, smem_u32(ar + G2_AT), P8, 8,
                         idesc_tf32_f32(128, 64), false);
        mma_panels<true>(tmem + 128, smem_u32(ar + G2_DWT), U16, smem_u32(ar + G2_AT), P8, 8,
                         idesc_tf32_f32(128, 64), false);
        mma_commit(&sm.bar_m[0]);
    }
    ok = ok && mbar_wait_bounded(&sm.bar_m[0], 0, kGradWait);
    if (tid == 0 && ok) {
        if (!direct) {
            // s dA^qk in rows 64..127 of [dR ; s dA^qk] and as its transposed rows
            mbar_arrive_expect_tx(&sm.bar_aq, 16384);
            bulk_g2s(ar + G2_DRQ + 8192, img + IM_AQ, 8192, &sm.bar_aq);
            bulk_g2s(ar + G2_DRQ + U16 + 8192, img + IM_AQ + 8192, 8192, &sm.bar_aq);
        } else {
            // the exact fp32 rows, where [dR ; s dA^qk] would be
            mbar_arrive_expect_tx(&sm.bar_aq, 16384);
            bulk_g2s(ar + G2_DRQ, img + IM_AQX, 16384, &sm.bar_aq);
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();

    // ---- step 2: dA^T-rows, A, the decayed operands ----
    if (quad < 2) {
        // lane = row i of dA; columns m = 32 hf ..
        float x[32];
        if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, hf * 32), x);
        else zero32(x);
        uint8_t *dst = ar + G2_DAT + (ch >> 5) * P8;
#pragma unroll
        for (int mm = 0; mm < 32; ++mm) f32_at(dst, i0 + mm, ch & 31) = tf32_operand(x[mm]);
    }
    {
        // A natural: row n holds A[n][m] over m
        const int n = tid >> 2, mb = (tid & 3) * 16;
        uint8_t *dst = ar + G2_AN + (mb >> 5) * P8;
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
            const int m = mb + 4 * e4;
            *reinterpret_cast<float4 *>(dst + sw128_chunk(n, (m & 31) >> 2)) =
                make_float4(f16_at(ar + G2_AF, n, m), f16_at(ar + G2_AF, n, m + 1),
                            f16_at(ar + G2_AF, n, m + 2), f16_at(ar + G2_AF, n, m + 3));
        }
    }
    if (!direct) {
        // K_hat^T (rows a, K = j) and [Q_tilde^T | K_tilde^T] (rows a, K = i)
        float kh[32], qt[32], kt[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const float kv = bfv(in.kp, ii), qv = bfv(in.xp, ii);
            const float ep = exp2_approx(in.G[ii] - Gm), en = exp2_approx(Gm - in.G[ii]);
            kh[ii] = kv * en;
            qt[ii] = qv * ep;
            kt[ii] = kv * ep;
        }
        row32_tf32(ar + G2_KH + hf * U16, ch, kh);
        row32_tf32(ar + G2_KQ + hf * U16, ch, qt);
        row32_tf32(ar + G2_KQ + (2 + hf) * U16, ch, kt);
    } else {
        // G, and k and q -- or, with block references, exp(G_r - G_i) k_i and
        // exp(G_i - G_r) q_i (r = the first token of i's 16-token block)
        float *gs = reinterpret_cast<float *>(ar + G2_GS), *ks = reinterpret_cast<float *>(ar + G2_KS),
              *qs = reinterpret_cast<float *>(ar + G2_QS);
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            const float gr = ii < 16 ? in.G[0] : in.G[16];
            gs[i * GD + ch] = in.G[ii];
            ks[i * GD + ch] = blocks ? exp2_approx(gr - in.G[ii]) * bfv(in.kp, ii) : bfv(in.kp, ii);
            qs[i * GD + ch] = blocks ? exp2_approx(in.G[ii] - gr) * bfv(in.xp, ii) : bfv(in.xp, ii);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        // (3) T1^T = dA^T A   (T1 = A^T dA; cols 192..255)
        mma_panels<true>(tmem + 192, smem_u32(ar + G2_DAT), P8, smem_u32(ar + G2_AT), P8, 8,
                         idesc_tf32_f32(128, 64), false);
        mma_commit(&sm.bar_m[1]);
    }
    ok = ok && mbar_wait_bounded(&sm.bar_m[1], 0, kGradWait);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();

    // ---- step 3: T1 (rows j) ----
    if (quad < 2) {
        // lane = m; columns j = 32 hf ..
        float x[32];
        if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, 192 + hf * 32), x);
        else zero32(x);
        uint8_t *dst = ar + G2_T1 + (ch >> 5) * P8;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) f32_at(dst, i0 + jj, ch & 31) = tf32_operand(x[jj]);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        // (4) -dR = T1 A^T   (cols 256..319)
        mma_panels<true>(tmem + 256, smem_u32(ar + G2_T1), P8, smem_u32(ar + G2_AN), P8, 8,
                         idesc_tf32_f32(128, 64), false);
        mma_commit(&sm.bar_m[2]);
    }
    ok = ok && mbar_wait_bounded(&sm.bar_m[2], 0, kGradWait);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();

    // ---- step 4: dR (strictly lower, rows i < L) into the decayed operands ----
    if (quad < 2) {
        // lane = row i of dR; columns n = 32 hf ..
        const int i = ch;
        float x[32];
        if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, 256 + hf * 32), x);
        else zero32(x);
#pragma unroll
        for (int nn = 0; nn < 32; ++nn) {
            const int n = i0 + nn;
            x[nn] = (n < i && i < L) ? -x[nn] : 0.f;
        }
        if (!direct) {
            row32_tf32(ar + G2_DRQ + hf * U16, i, x);
            uint8_t *drt = ar + G2_DRT + (i >> 5) * P8;  // rows n, K = i
            const float b = sm.beta[i];
#pragma unroll
            for (int nn = 0; nn < 32; ++nn) f32_at(drt, i0 + nn, i & 31) = tf32_operand(b * x[nn]);
        } else {
            // the direct path reads dR as plain fp32 rows
            float *drs = reinterpret_cast<float *>(ar + G2_DRT);
#pragma unroll
            for (int nn = 0; nn < 32; ++nn) drs[i * GC + i0 + nn] = x[nn];
        }
    }
    ok = ok && mbar_wait_bounded(&sm.bar_aq, 0, kGradWait);
    if (!direct) {
        // s dA^qk^T-rows (rows j, K = i) from rows 64.. of [dR ; s dA^qk]
        const int j = tid & 63, ib = (tid >> 6) * 16;
        uint8_t *src = ar + G2_DRQ + (j >> 5) * U16;
        uint8_t *dst = ar + G2_AQT + (ib >> 5) * P8;
#pragma unroll
        for (int e = 0; e < 16; ++e) f32_at(dst, j, (ib + e) & 31) = f32_at(src, 64 + ib + e, j & 31);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (!direct) {
        if (tid == 0 && ok) {
            tc_fence_after();
            // (5) [X1^T | X2^T] = K_hat^T [dR ; s dA^qk]^T   (cols 320..447)
            mma_panels<true>(tmem + 320, smem_u32(ar + G2_KH), U16, smem_u32(ar + G2_DRQ), U16, 8,
                             idesc_tf32_f32(128, 128), false);
            // (6) Y^T = Q_tilde^T (s dA^qk) + K_tilde^T Diag(beta) dR   (cols 448..511)
            mma_panels<true>(tmem + 448, smem_u32(ar + G2_KQ), U16, smem_u32(ar + G2_AQT), P8, 8,
                             idesc_tf32_f32(128, 64), false);
            mma_panels<true>(tmem + 448, smem_u32(ar + G2_KQ + 2 * U16), U16,
                             smem_u32(ar + G2_DRT), P8, 8, idesc_tf32_f32(128, 64), true);
            mma_commit(&sm.bar_m[3]);
        }
        ok = ok && mbar_wait_bounded(&sm.bar_m[3], 0, kGradWait);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
    } else if (blocks) {
        // Direct evaluation with 16-token block references (decays beyond
        // e^-80 across half a chunk, within 115 base 2 across each block):
        //   XR_i = sum_b exp(G_i - G_rb) sum_{j in b, j <= i} dR_ij [exp(G_rb - G_j) k_j]
        //   YY_j = sum_b exp(G_rb - G_j) sum_{i in b, i >= j}
        //              (beta_i dR_ij k_i + s dA^qk_ij q_i) exp(G_i - G_rb)
        // (r_b the first token of block b), so one 2^x per (row, block)
        // instead of one per (row, column); results straight into the same
        // TMEM columns as the split's products.
        const float *gs = reinterpret_cast<const float *>(ar + G2_GS);
        const float *kek = reinterpret_cast<const float *>(ar + G2_KS);
        const float *qp = reinterpret_cast<const float *>(ar + G2_QS);
        const float *drs = reinterpret_cast<const float *>(ar + G2_DRT);
        const float *das = reinterpret_cast<const float *>(ar + G2_DRQ);
        auto dr = [&](int i, int j) { return drs[i * GC + j]; };
        auto da = [&](int i, int j) { return das[i * GC + j]; };
        // beta_i exp(G_i - G_r) k_i into a dead operand area
        float *kp = reinterpret_cast<float *>(ar + G2_XS);
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            const float gr = ii < 16 ? in.G[0] : in.G[16];
            kp[i * GD + ch] = sm.beta[i] * exp2_approx(in.G[ii] - gr) * bfv(in.kp, ii);
        }
        __syncthreads();
        const uint32_t tl = tmem_addr(tmem, quad * 32, 0);
        // 4 rows (then 4 columns) of this thread's half at a time, inside one
        // block; dR and s dA^qk are zero outside their triangles, so whole
        // blocks are summed and rows of 4 columns load as float4
#pragma unroll 1
        for (int t4 = 0; t4 < 8; ++t4) {
            const int ib = i0 + 4 * t4, blk = ib >> 4;
            float gi[4], r[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 4; ++e) gi[e] = gs[(ib + e) * GD + ch];
            for (int b = 0; b <= blk; ++b) {
                const float gr = gs[(16 * b) * GD + ch];
                float rb[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
                for (int j = 16 * b; j < 16 * b + 16; j += 4) {
                    float w[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) w[c] = kek[(j + c) * GD + ch];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 x = *reinterpret_cast<const float4 *>(drs + (ib + e) * GC + j);
                        const float4 z = *reinterpret_cast<const float4 *>(das + (ib + e) * GC + j);
                        rb[e] = fmaf(x.x, w[0], fmaf(x.y, w[1], fmaf(x.z, w[2], fmaf(x.w, w[3], rb[e]))));
                        sb[e] = fmaf(z.x, w[0], fmaf(z.y, w[1], fmaf(z.z, w[2], fmaf(z.w, w[3], sb[e]))));
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float fb = exp2_approx(gi[e] - gr);
                    r[e] = fmaf(fb, rb[e], r[e]);
                    sq[e] = fmaf(fb, sb[e], sq[e]);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                tmem_st1_nowait(tl + 320 + hf * 32 + 4 * t4 + e, r[e]);
                tmem_st1_nowait(tl + 384 + hf * 32 + 4 * t4 + e, sq[e]);
            }
        }
#pragma unroll 1
        for (int t4 = 0; t4 < 8; ++t4) {
            const int jb = i0 + 4 * t4, blk = jb >> 4;
            float gj[4], y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 4; ++e) gj[e] = gs[(jb + e) * GD + ch];
            for (int b = blk; b < 4; ++b) {
                const float gr = gs[(16 * b) * GD + ch];
                float yb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int i = 16 * b; i < 16 * b + 16; ++i) {
                    const float kv = kp[i * GD + ch], qv = qp[i * GD + ch];
                    const float4 x = *reinterpret_cast<const float4 *>(drs + i * GC + jb);
                    const float4 z = *reinterpret_cast<const float4 *>(das + i * GC + jb);
                    yb[0] = fmaf(x.x, kv, fmaf(z.x, qv, yb[0]));
                    yb[1] = fmaf(x.y, kv, fmaf(z.y, qv, yb[1]));
                    yb[2] = fmaf(x.z, kv, fmaf(z.z, qv, yb[2]));
                    yb[3] = fmaf(x.w, kv, fmaf(z.w, qv, yb[3]));
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = fmaf(exp2_approx(gr - gj[e]), yb[e], y[e]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) tmem_st1_nowait(tl + 448 + hf * 32 + 4 * t4 + e, y[e]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    } else {
        // Direct evaluation (decays beyond e^-80 across half a chunk): every
        // exp(G_i - G_j) with i >= j (at most 1), into the same TMEM columns,
        // from dR and s dA^qk as fp32 rows.
        const float *gs = reinterpret_cast<const float *>(ar + G2_GS);
        const float *ks = reinterpret_cast<const float *>(ar + G2_KS);
        const float *qs = reinterpret_cast<const float *>(ar + G2_QS);
        const float *drs = reinterpret_cast<const float *>(ar + G2_DRT);
        const float *das = reinterpret_cast<const float *>(ar + G2_DRQ);
        auto dr = [&](int i, int j) { return drs[i * GC + j]; };
        auto da = [&](int i, int j) { return das[i * GC + j]; };
        // per-thread results go through a dead operand area (each thread
        // reads back only what it wrote)
        float *xrs = reinterpret_cast<float *>(ar + G2_XS), *xqs = xrs + GC * GD;
#pragma unroll 1
        for (int ii = 0; ii < 32; ++ii) {
            const int i = i0 + ii;
            const float gi = gs[i * GD + ch];
            float r = 0.f, s = 0.f;
            for (int j = 0; j <= i; ++j) {
                const float w = exp2_approx(gi - gs[j * GD + ch]) * ks[j * GD + ch];
                r = fmaf(dr(i, j), w, r);
                s = fmaf(da(i, j), w, s);
            }
            xrs[i * GD + ch] = r;
            xqs[i * GD + ch] = s;
        }
        float v[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) v[ii] = xrs[(i0 + ii) * GD + ch];
        tmem_st32(tmem_addr(tmem, quad * 32, 320 + hf * 32), v);
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) v[ii] = xqs[(i0 + ii) * GD + ch];
        tmem_st32(tmem_addr(tmem, quad * 32, 384 + hf * 32), v);
#pragma unroll 1
        for (int ii = 0; ii < 32; ++ii) {
            const int j = i0 + ii;
            const float gj = gs[j * GD + ch];
            float y = 0.f;
            for (int i = j; i < GC; ++i) {
                const float e = exp2_approx(gs[i * GD + ch] - gj);
                y = fmaf(sm.beta[i] * dr(i, j) * ks[i * GD + ch] + da(i, j) * qs[i * GD + ch], e,
                         y);
            }
            xrs[j * GD + ch] = y;
        }
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) v[ii] = xrs[(i0 + ii) * GD + ch];
        tmem_st32(tmem_addr(tmem, quad * 32, 448 + hf * 32), v);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // ---- epilogue: thread = channel ch (key, and value for dv), its tokens ----
    // dG per (token, channel) in shared memory for dlog_alpha's reverse sums;
    // dbeta's channel sums reduced across each warp's 32 channels first
    float *dgs = reinterpret_cast<float *>(ar + G2_DGS);
    float *pbs = reinterpret_cast<float *>(ar + G2_PS);  // [4 warp quadrants][64 tokens]
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int c0 = hf * 32 + g * 8;  // token / column offset of this group
        // dB2^T, dB1^T, XR, XQ, YY for the group's 8 tokens: one wait
        float y[5][8];
        const uint32_t tl = tmem_addr(tmem, quad * 32, c0);
        const uint32_t cols[5] = {tl + 128, tl + 64, tl + 320, tl + 384, tl + 448};
        if (ok) {
            tmem_ld8x5(cols, y);
        } else {
#pragma unroll
            for (int k = 0; k < 5; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) y[k][e] = 0.f;
        }
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int ii = g * 8 + e, i = c0 + e;
            const float b = sm.beta[i], gam = exp2_approx(in.G[ii]);
            const float kv = bfv(in.kp, ii);
            const float ep = direct ? 1.f : exp2_approx(in.G[ii] - Gm);
            const float en = direct ? 1.f : exp2_approx(Gm - in.G[ii]);
            // dB2 (B2 = Diag(beta)(exp(G) * K)), dB1 (B1 = Diag(beta) V, lane =
            // value channel), XR (rows of R), XQ (rows of A^qk), YY (columns of
            // R and A^qk)
            const float d2 = y[0][e], d1 = y[1][e], xr = ep * y[2][e], xq = ep * y[3][e],
                        yy = en * y[4][e];
            const float dkv = b * gam * d2 + b * xr + yy;
            float dgv = b * gam * kv * d2;
            dgv = fmaf(b * kv, xr, dgv);
            dgv = fmaf(bfv(in.xp, ii), xq, dgv);
            dgv = fmaf(-kv, yy, dgv);
            pv[e] = gam * kv * d2 + bfv(in.vp, ii) * d1 + kv * xr;
            if (i < L) {
                const size_t r = base + (size_t)i * rs;
                a.dv[r] = b * d1;
                atomicAdd(a.dq + r, xq);
                atomicAdd(a.dk + r, dkv);
            }
            dgs[i * GD + ch] = dgv;
        }
        // sum pv over the warp's 32 channels: halve the token set at each
        // exchange, then finish on one value; lane l ends with token
        // 4 (l>>4 & 1) + 2 (l>>3 & 1) + (l>>2 & 1) of the group
        const int lane = tid & 31;
        float w4[4], w2[2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const bool up = lane & 16;
            const float send = up ? pv[k] : pv[k + 4];
            w4[k] = (up ? pv[k + 4] : pv[k]) + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const bool up = lane & 8;
            const float send = up ? w4[k] : w4[k + 2];
            w2[k] = (up ? w4[k + 2] : w4[k]) + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        float z;
        {
            const bool up = lane & 4;
            z = (up ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, up ? w2[0] : w2[1], 4);
        }
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        if ((lane & 3) == 0)
            pbs[quad * GC + c0 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 +
                ((lane >> 2) & 1)] = z;
    }
    __syncthreads();
    {
        // this kernel's share of dlog_alpha: the reverse cumulative sum of its
        // dG, over each token half, then the second half's total onto the first
        float dg[32];
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) dg[ii] = dgs[(i0 + ii) * GD + ch];
        float acc = 0.f;
#pragma unroll
        for (int ii = 31; ii >= 0; --ii) {
            acc += dg[ii];
            dg[ii] = acc;
        }
        if (hf == 1) sm.gcarry[ch] = acc;  // the carries are read out: reuse
        if (tid >= GD && tid < GD + GC) {
            const int i = tid - GD;
            const float db = pbs[i] + pbs[GC + i] + pbs[2 * GC + i] + pbs[3 * GC + i];
            if (i < L) a.dbeta[(size_t)(t0 + i) * H + h] = db;
        }
        __syncthreads();
        const float add = hf == 0 ? sm.gcarry[ch] : 0.f;
#pragma unroll
        for (int ii = 0; ii < 32; ++ii)
            if (i0 + ii < L) atomicAdd(a.dlog_alpha + base + (size_t)(i0 + ii) * rs, dg[ii] + add);
    }
    const bool bad = __syncthreads_or(!ok);
    if (bad && tid == 0) {
        atomicExch(a.status, (int)KDA_ERR_TIMEOUT);
        (void)mbar_wait_bounded(&sm.bar_in, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_ld, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_aq, 0, kGradWait);
        (void)mbar_wait_bounded(&sm.bar_m[2], 0, kGradWait);
        if (!direct) (void)mbar_wait_bounded(&sm.bar_m[3], 0, kGradWait);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_chunk_grad(const ChunkGradArgs &a, cudaStream_t stream) {
    if (a.n_items == 0 || a.T == 0) return cudaSuccess;
    GradMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!encode_tile_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
        !encode_tile_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
        !encode_tile_map(&maps.v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
        !encode_tile_map(&maps.g, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H) ||
        (a.d_out &&
         !encode_tile_map(&maps.d, a.d_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H)))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_grad_g1_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kG1Smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_grad_g2_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kG2Smem);
    if (e != cudaSuccess) return e;
    chunk_grad_g1_kernel<<<(unsigned)a.n_items, kGThreads, kG1Smem, stream>>>(maps, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    chunk_grad_g2_kernel<<<(unsigned)a.n_items, kGThreads, kG2Smem, stream>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace kda
