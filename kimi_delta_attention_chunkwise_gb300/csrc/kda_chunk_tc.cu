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
// The engine regroups the last two lines (associativity only) so that the
// serial scan holds one matrix product per chunk:
//
//   M' = K_end^T W,  P' = K_end^T A^kk,  Q' = Q_hat - A^qk W,  Z = A^qk A^kk
//   S_c+1 = Diag(exp(G_last)) S_c + P' (beta V) - M' S_c
//   O     = Q' S_c + Z (beta V)
//
// Four launches on the caller's stream:
//   1. chunk_table  -- cu_seqlens -> first chunk index of every sequence
//                      (chunks restart at each sequence start).
//   2. chunk_prep   -- one CTA per (chunk, head), fully parallel: G, the
//                      decayed [K;Q] K^T products on the tensor core, the
//                      triangular solve, and W, M', P', Q', Z on the tensor
//                      core.  Writes f16 operand images (already in the
//                      128-byte-swizzled shared-memory layout) to scratch.
//   3. chunk_scan   -- one CTA per (sequence, head, 64-wide value tile):
//                      the only serial loop, over the chunks of a sequence.
//                      The fp32 state tile lives in registers; per chunk one
//                      dependent group of tcgen05 MMAs (-M' S_c, with
//                      P' (beta V) issued a chunk ahead), operands streamed
//                      in by a producer warp, and the state entering each
//                      chunk written out (f16) for the output pass.
//   4. chunk_out    -- one CTA per (chunk, head), fully parallel: the
//                      outputs from Q', Z, v and the stored states.
//
// Precision: every tensor-core product accumulates in fp32 (TMEM).  The
// decayed [K;Q] K^T product takes tf32 operands (the exp factors need fp32
// range); every other operand (A^kk, A^qk, W, K_end, M', P', Q', Z, beta V
// and the state S_c) is fp16, whose 11-bit significand keeps the result within
// the parity bound where bf16 operands (8 bits) do not.  The state itself
// stays fp32 in registers across the whole sequence.
//
// Overflow of the factorised decay (hard part of any tensor-core form): the
// products exp(G_i - G_j) are formed as exp(G_i - G_m) * exp(G_m - G_j) with
// the mid-chunk reference m, which is exact in fp32/bf16 range as long as
// |G_i - G_m| <= 80 for every channel and row.  A chunk that breaks this
// (decays stronger than ~exp(-80) across half a chunk) takes a CUDA-core path
// that evaluates every exp(G_i - G_j) directly, so any finite gates <= 0 work.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
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
// A decay factor exp(G_i - G_r) of the factorised products must stay within
// fp32 range: |G_i - G_r| <= 80, i.e. 80 log2(e) = 115.4 in the base-2 units
// the prep keeps G in.
constexpr float kSpanLimit2 = 115.f;

// Per-(chunk, head) scratch image: the scan's operands for one chunk, already
// in its shared-memory layout (f16, K-major, 128-byte swizzle), so the scan
// brings a chunk in with one bulk copy.  With
//   M' = K_end^T W        (128 x 128)   P' = K_end^T A^kk  (128 x 64)
//   Q' = Q_hat - A^qk W   (64 x 128)    Z  = A^qk A^kk     (64 x 64)
// the chunk's recurrence and outputs are
//   S_c+1 = Diag(Gamma_last) S_c + P' (beta V) - M' S_c
//   O     = Q' S_c + Z (beta V)
// (K_end^T E and A^qk E with E = U - W S_c, U = A^kk beta V, expanded).
constexpr uint32_t IMG_MN = 0;          // -M': 2 panels of 128 rows
constexpr uint32_t IMG_P = 32768;       // P' : 128 rows
constexpr uint32_t IMG_Q0 = 49152;      // Q' keys 0..63  : 64 rows
constexpr uint32_t IMG_Z = 57344;       // Z  : 64 rows
constexpr uint32_t IMG_Q1 = 65536;      // Q' keys 64..127: 64 rows
constexpr uint32_t IMG_GB = 73728;      // Gamma_last [128] f32, beta [64] f32
constexpr uint32_t IMG_BYTES = IMG_GB + 768;   // bytes written per chunk (the scan
                                               // copies the operands, IMG_GB bytes)
constexpr uint32_t IMG_STRIDE = 74752;         // 73 KB slot, 1024-aligned
static_assert(IMG_BYTES <= IMG_STRIDE && IMG_STRIDE % 1024 == 0, "image slot");
// As 128-row MMA A operands the 64-row tiles are read with the 8 KB that
// precedes them: rows 64..127 of [filler ; Q'] and [filler ; Z] hold them, and
// the filler rows produce accumulator rows that are never read.

struct Scratch {
    uint8_t *img;        // [n_chunks x H] x IMG_STRIDE
    uint8_t *sst;        // [n_chunks x H x value tiles] S_c images (f16, 16 KB each)
    uint32_t *ready;     // image written [n_chunks x H], then state images written
                         // [n_chunks x H x value tiles] (kernels run concurrently)
    int2 *chunk_tok;     // [max chunks] first token and length of each chunk (0: none)
    int32_t *chunk_off;  // [N + 1]
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t max_chunks(int32_t N, int32_t T) {
    return (size_t)T / C + (size_t)N + 1;
}

Scratch carve(void *ws, int32_t N, int32_t T, int32_t H) {
    const size_t nch = max_chunks(N, T) * (size_t)H;
    uint8_t *p = static_cast<uint8_t *>(ws);
    Scratch s;
    s.img = p; p += align256(nch * IMG_STRIDE);
    s.sst = p; p += align256(nch * NT * (size_t)(D * 128));
    s.ready = reinterpret_cast<uint32_t *>(p); p += align256(nch * (1 + NT) * sizeof(uint32_t));
    s.chunk_tok = reinterpret_cast<int2 *>(p); p += align256(max_chunks(N, T) * sizeof(int2));
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
// 1. chunk table (CTA 0): chunk_off[s] = number of chunks before sequence s,
//    and chunk_tok[c] = {first token, length} of chunk c ({0, 0} past the
//    last chunk); every CTA also clears a share of the n_ready image and
//    state flags.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t *cu, int32_t N,
                                                           int32_t T, int32_t *chunk_off,
                                                           int2 *chunk_tok, uint32_t *ready,
                                                           size_t n_ready) {
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();  // the next kernel waits for this one's results
    for (size_t i = (size_t)blockIdx.x * 1024 + tid; i < n_ready; i += (size_t)gridDim.x * 1024)
        ready[i] = 0u;
    if (blockIdx.x != 0) return;
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
    __syncthreads();  // chunk_off is visible to the whole CTA
    const int32_t total = chunk_off[N], n_max = (int32_t)max_chunks(N, T);
    for (int32_t c = tid; c < n_max; c += 1024) {
        int2 tok = make_int2(0, 0);
        if (c < total) {
            const int32_t s = find_seq(chunk_off, N, c);
            int32_t a, b;
            seq_bounds(cu, s, T, a, b);
            tok.x = a + (c - chunk_off[s]) * C;
            tok.y = min(C, b - tok.x);
        }
        chunk_tok[c] = tok;
    }
}


// ---------------------------------------------------------------------------
// 2. per-(chunk, head) preparation: a persistent kernel
// ---------------------------------------------------------------------------
// One CTA per SM it runs on, holding two independent workers of 256 threads
// (each with its own shared memory, mbarriers, named barrier and 256 TMEM
// columns).  Worker w of W takes items (chunk, head) w, w + W, w + 2W, ...
// -- heads fastest, the order in which the scan consumes the images; w runs
// over the CTAs first, so a partial last round spreads over the SMs.  A
// kernel launched after this one starts only once every CTA of this grid is
// running, so it may wait on any item's image: the item's worker is running.
// A worker's image stores drain while its next item's tiles load: thread 0
// waits for them (and publishes the flag) only after issuing those loads.
//
// Within a worker, thread t owns key channel d = t % 128 for the tokens of
// one half chunk (t / 128).  Shared memory, with regions reused once their
// first tenant is done:
//   a1: g tile (TMA, f32 [64][128]) -> tf32 [K_tilde ; Q_tilde], 128 rows x
//       128 K in 4 panels (64 KB) -> R, X (= A^kk) and the solve's block
//       products (fp32), with A^qk and K_end^T (f16, at kOffAqk, kOffKe) kept
//       beside them -> W^T (f16, at 0) -> the staging of the image's -M', P'
//       and Q' panels, in image order;
//   b1: k and q tiles (TMA, bf16 [64][128] each) -> tf32 K_hat, 64 rows x
//       128 K in 4 panels (32 KB) (direct path: G f32 [64][128]) -> A^kk and
//       A^kk^T (f16, 8 KB each) and (beta Gamma K)^T (f16, 128 x 64, 16 KB)
//       -> Z staging (at 0).
// TMEM (fp32, lane = row): cols 0..63 the decayed products; 64..95 the half
// path's cross block; 96..159 (beta Gamma K)^T and K_end^T as f16 pairs,
// parked while the first products still read their operand slots; 160..191
// the half path's K_hat about token 48, likewise; 192..255 -Q_hat^T.  Then
// Z (0..63) and W^T (64..127); then M' (0..127), P' (128..191) and -Q'^T
// (192..255, accumulated onto -Q_hat^T).
//
// The decayed products exp(G_i - G_j) (j <= i, so at most 1) are split as
// exp(G_i - G_r) * exp(G_r - G_j) about a reference token r, in one of three
// ways per item:
//   mid   -- r = 32 for the whole chunk, when every |G_i - G_32| <= 80: one
//            tf32 MMA [K_tilde ; Q_tilde] K_hat^T;
//   half  -- r = 16 for the first half's rows and columns, r = 48 for the
//            second's, when every |G_i - G_r| <= 80 within its half (log
//            decays down to -5 per token, the K3 gate's range): the same MMA
//            gives both diagonal half blocks; the block of second-half rows
//            and first-half columns comes from a second MMA whose B operand
//            is K_hat about r = 48 for the first half's tokens (exponent
//            G_48 - G_j <= 0);
//   direct-- every exp(G_i - G_j) on CUDA cores (decays stronger than e^-80
//            within a quarter chunk).
constexpr int kPrepWorkerThreads = 256;
constexpr int kPrepWorkers = 2;
constexpr int kPrepThreads = kPrepWorkerThreads * kPrepWorkers;
constexpr int HALF = C / 2;

struct PrepSmem {
    uint8_t a1[4 * 16384];
    uint8_t b1[4 * 8192];
    float beta[C];
    // cumulative log decays in base 2 (G log2 e) of each channel at:
    float gcarry[D];   // token 31
    float gmid[D];     // the reference token MID
    float gh1[D];      // token 48 (the second half's reference)
    float glast[D];    // the chunk's last token
    float knorm[C];    // 1 / |k_i|, 1 / |q_i| (L2 prologue; else 1)
    float qnorm[C];
    uint64_t bar_in, bar_mma;
    uint64_t published;  // thread 0: the item whose image flag is still to go up (~0: none)
    uint32_t n_path[3];  // items per decay path (thread 0)
};
constexpr size_t kPrepWorkerBytes = (sizeof(PrepSmem) + 1023) & ~size_t(1023);
// R and X rows are kRS floats apart (a multiple of 4: rows load as float4;
// 68 = 4 mod 32 keeps the column reads of the transposed A^kk store at most
// two-way bank conflicted); the block products Tb rows kTS floats apart.
constexpr int kRS = C + 4;
constexpr int kTS = 34;
constexpr uint32_t kOffX = C * kRS * 4;            // X after R inside a1
constexpr uint32_t kOffTb = 2 * C * kRS * 4;       // block products after X
constexpr uint32_t kOffAqk = 40960;                // A^qk (f16) inside a1
constexpr uint32_t kOffKe = 49152;                 // K_end^T (f16) inside a1
constexpr uint32_t kOffAkT = 8192;                 // A^kk^T after A^kk inside b1
constexpr uint32_t kOffA2 = 16384;                 // (beta Gamma K)^T inside b1
static_assert(kOffTb + 32 * kTS * 4 <= kOffAqk, "solve scratch below A^qk");
constexpr uint32_t kInBytes = 2 * C * D * 2 + C * D * 4;  // k, q bf16 + g f32 tiles
static_assert(kOffTb + 32 * kTS * 4 <= 4 * 16384, "a1 reuse");
static_assert(kOffX % 16 == 0 && kOffTb % 16 == 0 && kRS % 4 == 0 && kTS % 2 == 0,
              "vector access to R, X and Tb");
static_assert(MID == HALF, "the reference token opens the second half");

// Named barrier over one worker's 256 threads (ids 1 and 2; 0 is the CTA's),
// with the id as an immediate (a warp-uniform branch picks it).
template <int ID>
__device__ __forceinline__ void wbar_id() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(kPrepWorkerThreads) : "memory");
}
__device__ __forceinline__ void wbar(int id) {
    if (id == 1) wbar_id<1>();
    else wbar_id<2>();
}
// The same barrier, returning the OR of a predicate over the worker.
template <int ID>
__device__ __forceinline__ bool wbar_or_id(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(ID), "n"(kPrepWorkerThreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool wbar_or(int id, bool pred) {
    return id == 1 ? wbar_or_id<1>(pred) : wbar_or_id<2>(pred);
}

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

// The inverse of a unit lower-triangular L = I + R, two levels up from its
// 16 x 16 diagonal-block inverses.  For a split L = [A 0; B D] with A and D
// square, L^-1 = [A^-1 0; -D^-1 B A^-1  D^-1].  Level 1 applies it inside the
// two 32 x 32 diagonal blocks (16 x 16 halves), level 2 to the whole 64 x 64
// (32 x 32 halves); B is the block of R below the diagonal.  The products run
// over full K ranges: X is zero above its diagonal.  One worker (256 threads).
__device__ __forceinline__ void solve_level16(float (*R)[kRS], float (*X)[kRS],
                                              float (*Tb)[kTS], int tid, int bid) {
    // thread -> 32 x 32 block p, one row of its lower-left 16 x 16, two columns
    const int p = tid >> 7, t = tid & 127, o = 32 * p;
    const int lr = t >> 3, lc = (t & 7) * 2;
    const int r = o + 16 + lr, c = o + lc;
    float a0 = 0.f, a1 = 0.f;  // (B A^-1)[r][c]
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
        const float4 rv = *reinterpret_cast<const float4 *>(&R[r][o + 4 * k4]);
        const float rs[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 xv = *reinterpret_cast<const float2 *>(&X[o + 4 * k4 + e][c]);
            a0 = fmaf(rs[e], xv.x, a0);
            a1 = fmaf(rs[e], xv.y, a1);
        }
    }
    *reinterpret_cast<float2 *>(&Tb[16 * p + lr][lc]) = make_float2(a0, a1);
    wbar(bid);
    float b0 = 0.f, b1 = 0.f;  // (D^-1 B A^-1)[r][c]
#pragma unroll
    for (int m4 = 0; m4 < 4; ++m4) {
        const float4 xv = *reinterpret_cast<const float4 *>(&X[r][o + 16 + 4 * m4]);
        const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 tv = *reinterpret_cast<const float2 *>(&Tb[16 * p + 4 * m4 + e][lc]);
            b0 = fmaf(xs[e], tv.x, b0);
            b1 = fmaf(xs[e], tv.y, b1);
        }
    }
    *reinterpret_cast<float2 *>(&X[r][c]) = make_float2(-b0, -b1);
    wbar(bid);
}
__device__ __forceinline__ void solve_level32(float (*R)[kRS], float (*X)[kRS],
                                              float (*Tb)[kTS], int tid, int bid) {
    // thread -> 2 x 2 tile of the lower-left 32 x 32: rows 32 + rr.., columns cc..
    const int rr = (tid >> 4) * 2, cc = (tid & 15) * 2, r = 32 + rr;
    float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;  // B A^-1
#pragma unroll 4
    for (int k4 = 0; k4 < 8; ++k4) {
        const float4 ra = *reinterpret_cast<const float4 *>(&R[r][4 * k4]);
        const float4 rb = *reinterpret_cast<const float4 *>(&R[r + 1][4 * k4]);
        const float as[4] = {ra.x, ra.y, ra.z, ra.w}, bs[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 xv = *reinterpret_cast<const float2 *>(&X[4 * k4 + e][cc]);
            a00 = fmaf(as[e], xv.x, a00);
            a01 = fmaf(as[e], xv.y, a01);
            a10 = fmaf(bs[e], xv.x, a10);
            a11 = fmaf(bs[e], xv.y, a11);
        }
    }
    *reinterpret_cast<float2 *>(&Tb[rr][cc]) = make_float2(a00, a01);
    *reinterpret_cast<float2 *>(&Tb[rr + 1][cc]) = make_float2(a10, a11);
    wbar(bid);
    float b00 = 0.f, b01 = 0.f, b10 = 0.f, b11 = 0.f;  // D^-1 B A^-1
#pragma unroll 4
    for (int m4 = 0; m4 < 8; ++m4) {
        const float4 xa = *reinterpret_cast<const float4 *>(&X[r][32 + 4 * m4]);
        const float4 xb = *reinterpret_cast<const float4 *>(&X[r + 1][32 + 4 * m4]);
        const float as[4] = {xa.x, xa.y, xa.z, xa.w}, bs[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 tv = *reinterpret_cast<const float2 *>(&Tb[4 * m4 + e][cc]);
            b00 = fmaf(as[e], tv.x, b00);
            b01 = fmaf(as[e], tv.y, b01);
            b10 = fmaf(bs[e], tv.x, b10);
            b11 = fmaf(bs[e], tv.y, b11);
        }
    }
    *reinterpret_cast<float2 *>(&X[r][cc]) = make_float2(-b00, -b01);
    *reinterpret_cast<float2 *>(&X[r + 1][cc]) = make_float2(-b10, -b11);
    wbar(bid);
}

struct PrepMaps {
    CUtensorMap q, k, g;  // [T, H, D] viewed as {D, H, T}, box {128, 1, 64}
};

// Items of each path for the decayed products (mid, half, direct), per device;
// kda_chunk_path_counts() reads and clears them.
__device__ unsigned long long g_path_counts[3];

// PRO: the kernel applies an input prologue (compiled out when false)
template <bool PRO>
__global__ void __launch_bounds__(kPrepThreads, 1)
chunk_prep_kernel(const __grid_constant__ PrepMaps maps, const __nv_bfloat16 *__restrict__ q,
                  const __nv_bfloat16 *__restrict__ k, const float *__restrict__ beta,
                  float scale, int32_t H, int32_t grp, int32_t pro,
                  const float *__restrict__ gbias, const float *__restrict__ galog, Scratch sc,
                  uint32_t n_items, int32_t flags, long long wait_cycles, int *status,
                  uint8_t *__restrict__ bwd_aux) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int wk = threadIdx.x / kPrepWorkerThreads;
    PrepSmem &sm = *reinterpret_cast<PrepSmem *>(base + wk * kPrepWorkerBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kPrepWorkers * kPrepWorkerBytes);
    float(*R)[kRS] = reinterpret_cast<float(*)[kRS]>(sm.a1);
    float(*X)[kRS] = reinterpret_cast<float(*)[kRS]>(sm.a1 + kOffX);
    float(*Tb)[kTS] = reinterpret_cast<float(*)[kTS]>(sm.a1 + kOffTb);
    uint8_t *b2 = sm.b1;              // A^kk, f16 panel
    uint8_t *akt = sm.b1 + kOffAkT;   // A^kk^T, f16 panel
    uint8_t *a2 = sm.b1 + kOffA2;     // (beta Gamma K)^T, f16 panel
    uint8_t *aqk = sm.a1 + kOffAqk;   // A^qk, f16 panel
    uint8_t *ket = sm.a1 + kOffKe;    // K_end^T, f16 panel
    uint8_t *wt = sm.a1;              // W^T, f16 panel (after the solve)
    uint8_t *zst = sm.b1;             // Z staging (after the MMAs that read A^kk)

    const int tid = threadIdx.x % kPrepWorkerThreads, warp = tid >> 5, lane = tid & 31;
    const int bid = 1 + wk;           // the worker's named barrier
    // The chunk table (and the cleared flags) first; then the
    // next kernel may start: it only waits on items of this running grid.
    pdl_wait_primaries();
    pdl_launch_dependents();
    if (tid == 0) {
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
        sm.n_path[0] = sm.n_path[1] = sm.n_path[2] = 0u;
        sm.published = ~0ull;
    }
    if (threadIdx.x < 32) {
        tmem_alloc(tmem_slot, 256 * kPrepWorkers);  // both workers' columns at once
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot + (uint32_t)wk * 256u;
    const uint32_t stride = gridDim.x * (uint32_t)kPrepWorkers;  // items between a worker's own
    const int d = tid & (D - 1), hf = tid >> 7, i0 = hf * HALF;
    const bool l2 = PRO && (pro & KDA_PROLOGUE_L2NORM_QK);
    const bool gate = PRO && (pro & KDA_PROLOGUE_GATE);
    uint32_t in_phase = 0, mma_phase = 0;
    bool ok = true;

    for (uint32_t item = (uint32_t)wk * gridDim.x + blockIdx.x; item < n_items;
         item += stride) {
        const int32_t c = (int32_t)(item / (uint32_t)H), h = (int32_t)(item % (uint32_t)H);
        const int2 tok = sc.chunk_tok[c];
        const int32_t t0 = tok.x, L = tok.y;
        if (L <= 0) break;  // past the last chunk: so is every later item
        const size_t ch = (size_t)c * H + h;
        uint8_t *img = sc.img + ch * IMG_STRIDE;
        float *gb = reinterpret_cast<float *>(img + IMG_GB);
        const int32_t hq = h / grp;                 // the q/k head of this value head's group
        const size_t rs = (size_t)(H / grp) * D;    // q/k token stride

        // Stream the chunk's k, q and log-decay tiles in (one tensor load each),
        // once the previous item's first group of image stores (-M' from a1,
        // Z from b1) has left shared memory; its second group reads the upper
        // half of a1, which the tiles do not touch.
        if (tid == 0) {
            bulk_wait_group_read<1>();
            mbar_arrive_expect_tx(&sm.bar_in, kInBytes);
            tma_load_3d(sm.b1, &maps.k, 0, hq, t0, &sm.bar_in);
            tma_load_3d(sm.b1 + C * D * 2, &maps.q, 0, hq, t0, &sm.bar_in);
            tma_load_3d(sm.a1, &maps.g, 0, h, t0, &sm.bar_in);
            // the previous image out of shared memory (its upper half is
            // rewritten below) and, with flags, complete in global memory:
            // publish it
            if (flags) bulk_wait_group_all();
            else bulk_wait_group_read<0>();
            if (flags && sm.published != ~0ull) {
                fence_proxy_async_global();
                flag_release(sc.ready + sm.published, 1u);
            }
            sm.published = ~0ull;
        } else if (tid == 32) {
            // this worker's next item goes to L2 early
            const uint32_t ahead = item + stride;
            if (ahead < n_items) {
                const int32_t ca = (int32_t)(ahead / (uint32_t)H),
                              ha = (int32_t)(ahead % (uint32_t)H);
                const int2 ta = sc.chunk_tok[ca];
                if (ta.y > 0) {
                    tma_prefetch_l2_3d(&maps.k, 0, ha / grp, ta.x);
                    tma_prefetch_l2_3d(&maps.q, 0, ha / grp, ta.x);
                    tma_prefetch_l2_3d(&maps.g, 0, ha, ta.x);
                }
            }
        }
        // beta: loaded now, stored once the tiles are in (its latency hides under theirs)
        float beta_i = 0.f;
        if (tid < C && tid < L) beta_i = beta[(size_t)(t0 + tid) * H + h];
        const float sens = gate ? __expf(galog[h]) : 0.f;
        const float gbias_d = gate ? gbias[(size_t)h * D + d] : 0.f;
        ok = mbar_wait_bounded(&sm.bar_in, in_phase, wait_cycles) && ok;
        in_phase ^= 1u;
        if (tid < C) {
            if (PRO && (pro & KDA_PROLOGUE_BETA_LOGITS) && tid < L) beta_i = pro_sigmoid(beta_i);
            sm.beta[tid] = beta_i;  // read after the next worker barrier
            gb[128 + tid] = beta_i;
        }

        uint32_t kp[HALF / 2], qp[HALF / 2];
        float G[HALF];  // cumulative log decay of this thread's tokens, base 2 (G log2 e)
        {
            const float *gs = reinterpret_cast<const float *>(sm.a1);
            unsigned short *ks = reinterpret_cast<unsigned short *>(sm.b1);
            unsigned short *qs = ks + C * D;
            // The L2 prologue, on the tiles in shared memory: warp w finds 1/|k_i|
            // and 1/|q_i| of tokens 8w .. 8w + 7 and rescales their rows in place
            // as fp16 (11-bit significand: the tf32 and fp16 operands built from
            // them keep their precision; bf16 here cost a visible share of the
            // error budget).  The stored inverse norms serve the direct path,
            // which reads the raw rows from global memory.
            if (l2) {
#pragma unroll 1
                for (int i = warp * 8; i < warp * 8 + 8; ++i) {
                    uint2 *kr = reinterpret_cast<uint2 *>(ks + i * D + lane * 4);
                    uint2 *qr = reinterpret_cast<uint2 *>(qs + i * D + lane * 4);
                    const uint2 kw = *kr, qw = *qr;
                    const uint32_t kv4[2] = {kw.x, kw.y}, qv4[2] = {qw.x, qw.y};
                    float kf[4], qf[4], kk = 0.f, qq = 0.f;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        kf[2 * e] = __uint_as_float(kv4[e] << 16);
                        kf[2 * e + 1] = __uint_as_float(kv4[e] & 0xFFFF0000u);
                        qf[2 * e] = __uint_as_float(qv4[e] << 16);
                        qf[2 * e + 1] = __uint_as_float(qv4[e] & 0xFFFF0000u);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kk = fmaf(kf[e], kf[e], kk);
                        qq = fmaf(qf[e], qf[e], qq);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        kk += __shfl_xor_sync(0xffffffffu, kk, o);
                        qq += __shfl_xor_sync(0xffffffffu, qq, o);
                    }
                    const float rk = rsqrtf(kk + kL2Eps), rq = rsqrtf(qq + kL2Eps);
                    *kr = make_uint2(pack_f16x2(kf[0] * rk, kf[1] * rk),
                                     pack_f16x2(kf[2] * rk, kf[3] * rk));
                    *qr = make_uint2(pack_f16x2(qf[0] * rq, qf[1] * rq),
                                     pack_f16x2(qf[2] * rq, qf[3] * rq));
                    if (lane == 0) {
                        sm.knorm[i] = rk;
                        sm.qnorm[i] = rq;
                    }
                }
                wbar(bid);
            }
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
                float lg = (i0 + ii < L) ? gs[(i0 + ii) * D + d] : 0.f;
                if (gate && i0 + ii < L) lg = pro_gate(lg, sens, gbias_d);
                acc = fmaf(lg, kLog2e, acc);
                G[ii] = acc;
            }
        }
        if (hf == 0) sm.gcarry[d] = G[HALF - 1];
        wbar(bid);  // staging consumed; carries published
        if (hf == 1) {
            const float carry = sm.gcarry[d];
#pragma unroll
            for (int ii = 0; ii < HALF; ++ii) G[ii] += carry;
            sm.gmid[d] = G[0];
            sm.gh1[d] = G[HALF / 2];
            sm.glast[d] = G[HALF - 1];
        }
        wbar(bid);
        const float Gm = sm.gmid[d], Gl = sm.glast[d];
        // the path: mid reference if it stays in range, else one per half, else direct
        const float Gh = G[HALF / 2];  // this half's reference token (16 or 48)
        float span = 0.f;
#pragma unroll
        for (int ii = 0; ii < HALF; ++ii) span = fmaxf(span, fabsf(G[ii] - Gm));
        int path = wbar_or(bid, !(span <= kSpanLimit2)) ? 1 : 0;
        if (path) {
            span = 0.f;
#pragma unroll
            for (int ii = 0; ii < HALF; ++ii) span = fmaxf(span, fabsf(G[ii] - Gh));
            path = wbar_or(bid, !(span <= kSpanLimit2)) ? 2 : 1;
        }
        if (tid == 0) ++sm.n_path[path];
        const float Gr = path == 1 ? Gh : Gm;  // reference of this thread's tokens
        // k and q of this thread's tokens: bf16 inputs, or fp16 once the L2
        // prologue has normalised them
        auto unpack = [&](uint32_t w, int hi) {
            if (l2)
                return __half2float(
                    __ushort_as_half((unsigned short)(hi ? (w >> 16) : (w & 0xFFFFu))));
            return __uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16));
        };
        auto kval = [&](int ii) { return unpack(kp[ii >> 1], ii & 1); };
        auto qval = [&](int ii) { return unpack(qp[ii >> 1], ii & 1); };

        if (path == 2) {
            // Direct path: every exp(G_i - G_j) taken directly (exponent <= 0).
            float *Gs = reinterpret_cast<float *>(sm.b1);  // [64][128]
#pragma unroll
            for (int ii = 0; ii < HALF; ++ii) Gs[(i0 + ii) * D + d] = G[ii];
            wbar(bid);
            const __nv_bfloat16 *kc = k + ((size_t)t0 * (H / grp) + hq) * D;
            const __nv_bfloat16 *qc = q + ((size_t)t0 * (H / grp) + hq) * D;
            for (int i = warp; i < C; i += kPrepWorkerThreads / 32) {
                for (int j = 0; j <= i; ++j) {
                    float r = 0.f, a = 0.f;
                    if (i < L) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const int dd = lane + 32 * m;
                            const float w = exp2_approx(Gs[i * D + dd] - Gs[j * D + dd]) *
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
                        // the L2 prologue rescales the raw dot products
                        const float nk = l2 ? sm.knorm[i] * sm.knorm[j] : 1.f;
                        const float nq = l2 ? sm.qnorm[i] * sm.knorm[j] : 1.f;
                        R[i][j] = (j < i) ? sm.beta[i] * r * nk : 0.f;
                        X[i][j] = scale * a * nq;
                    }
                }
                for (int j = i + 1 + lane; j < C; j += 32) {
                    R[i][j] = 0.f;
                    X[i][j] = 0.f;
                }
            }
            wbar(bid);
            if (tid < C) {
                float row[64];
#pragma unroll
                for (int j = 0; j < 64; ++j) row[j] = X[tid][j];
                store_row_f16_image(aqk, tid, row);
            }
            wbar(bid);
            // The direct path's last uses of G, k and q (the tf32 paths made them
            // while building their operands): -Q_hat^T (Q_hat_i = s Gamma_i q_i)
            // into TMEM cols 192..255 (lane d, token columns), where the last MMA
            // group adds (A^qk W)^T to give -Q'^T; (beta Gamma K)^T and K_end^T (row
            // d, this thread's half of the tokens, f16) into their operand slots.
            {
                float row[32];
#pragma unroll
                for (int ii = 0; ii < HALF; ++ii)
                    row[ii] = -scale * exp2_approx(G[ii]) * qval(ii);
                tmem_st32(tmem_addr(tmem, (warp & 3) * 32, 192 + hf * 32), row);
#pragma unroll
                for (int ii = 0; ii < HALF; ++ii)
                    row[ii] = sm.beta[i0 + ii] * exp2_approx(G[ii]) * kval(ii);
                store_quarter_f16_image(a2, d, hf * 4, row);
#pragma unroll
                for (int ii = 0; ii < HALF; ++ii) row[ii] = exp2_approx(Gl - G[ii]) * kval(ii);
                store_quarter_f16_image(ket, d, hf * 4, row);
            }
        } else {
            // The decay-factorised tf32 operands, token by token.
            // With them, the last uses of G, k and q, so that they leave the
            // registers here: -Q_hat^T (Q_hat_i = s Gamma_i q_i) into TMEM cols
            // 192..255 (lane d, token columns), where the last MMA group adds
            // (A^qk W)^T to give -Q'^T; (beta Gamma K)^T and K_end^T as f16 pairs
            // into TMEM cols 96..159 until the products free their operand slots
            // (per 8 tokens: 4 columns of beta Gamma K, then 4 of K_end).
            const uint32_t pa = (d >> 5) * 16384u, pb = (d >> 5) * 8192u;
            const uint32_t tl = tmem_addr(tmem, (warp & 3) * 32, 0);
#pragma unroll
            for (int g8 = 0; g8 < HALF / 8; ++g8) {
                uint32_t qh[8], pk[8];
                float bk0 = 0.f, ke0 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int ii = g8 * 8 + e, i = i0 + ii;
                    const float kv = kval(ii), qv = qval(ii);
                    const float ep = exp2_approx(G[ii] - Gr), en = exp2_approx(Gr - G[ii]);
                    *reinterpret_cast<float *>(sm.a1 + pa + sw128_offset_f32(i, d & 31)) =
                        tf32_operand(kv * ep);
                    *reinterpret_cast<float *>(sm.a1 + pa + sw128_offset_f32(64 + i, d & 31)) =
                        tf32_operand(qv * ep);
                    *reinterpret_cast<float *>(sm.b1 + pb + sw128_offset_f32(i, d & 31)) =
                        tf32_operand(kv * en);
                    const float gam = exp2_approx(G[ii]);
                    const float bk = sm.beta[i] * gam * kv, ke = exp2_approx(Gl - G[ii]) * kv;
                    qh[e] = __float_as_uint(-scale * gam * qv);
                    if (e & 1) {
                        pk[e >> 1] = pack_f16x2(bk0, bk);
                        pk[4 + (e >> 1)] = pack_f16x2(ke0, ke);
                    } else {
                        bk0 = bk;
                        ke0 = ke;
                    }
                }
                tmem_st8_nowait(tl + 192 + hf * 32 + g8 * 8, qh);
                tmem_st8_nowait(tl + 96 + hf * 32 + g8 * 8, pk);
                if (path == 1 && hf == 0) {
                    // the half path's K_hat about token 48 for tokens 0..31
                    // (exponents G_48 - G_j <= 0), parked in cols 160..191
                    const float G48 = sm.gh1[d];
                    uint32_t kh[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int ii = g8 * 8 + e;
                        kh[e] = __float_as_uint(
                            tf32_operand(kval(ii) * exp2_approx(G48 - G[ii])));
                    }
                    tmem_st8_nowait(tl + 160 + g8 * 8, kh);
                }
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            wbar(bid);
            // [K_tilde ; Q_tilde] K_hat^T on the tensor core (tf32): TMEM cols 0..63.
            if (tid == 0 && ok) {
                tc_fence_after();
                mma_panels<true>(tmem, smem_u32(sm.a1), 16384, smem_u32(sm.b1), 8192, 16,
                                 idesc_tf32_f32(128, 64), false);
                mma_commit(&sm.bar_mma);
            }
            if (ok) ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, wait_cycles);
            mma_phase ^= 1u;
            if (path == 1) {
                // Second-half rows, first-half columns: K_hat about token 48 for
                // tokens 0..31 (parked in TMEM above) over the consumed K_hat rows
                // 0..31, then A (still intact) times it into TMEM cols 64..95.
                tc_fence_after();
                if (hf == 0) {
                    float kh[32];
                    if (ok) {
                        tmem_ld32(tmem_addr(tmem, (warp & 3) * 32, 160), kh);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) kh[j] = 0.f;
                    }
#pragma unroll
                    for (int ii = 0; ii < HALF; ++ii)
                        *reinterpret_cast<float *>(sm.b1 + pb + sw128_offset_f32(ii, d & 31)) =
                            kh[ii];
                }
                fence_proxy_async();
                tc_fence_before();
                wbar(bid);
                if (tid == 0 && ok) {
                    tc_fence_after();
                    mma_panels<true>(tmem + 64, smem_u32(sm.a1), 16384, smem_u32(sm.b1), 8192,
                                     16, idesc_tf32_f32(128, 32), false);
                    mma_commit(&sm.bar_mma);
                }
                if (ok) ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, wait_cycles);
                mma_phase ^= 1u;
            }
            ok = __all_sync(0xffffffffu, ok);  // TMEM loads below are warp-collective
            tc_fence_after();
            {
                // the parked (beta Gamma K)^T and K_end^T into their operand
                // slots, which the products have consumed
                float pv[32];
                if (ok) {
                    tmem_ld32(tmem_addr(tmem, (warp & 3) * 32, 96 + hf * 32), pv);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) pv[j] = 0.f;
                }
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    *reinterpret_cast<uint4 *>(a2 + sw128_chunk(d, hf * 4 + g8)) =
                        make_uint4(__float_as_uint(pv[g8 * 8 + 0]), __float_as_uint(pv[g8 * 8 + 1]),
                                   __float_as_uint(pv[g8 * 8 + 2]), __float_as_uint(pv[g8 * 8 + 3]));
                    *reinterpret_cast<uint4 *>(ket + sw128_chunk(d, hf * 4 + g8)) =
                        make_uint4(__float_as_uint(pv[g8 * 8 + 4]), __float_as_uint(pv[g8 * 8 + 5]),
                                   __float_as_uint(pv[g8 * 8 + 6]), __float_as_uint(pv[g8 * 8 + 7]));
                }
            }
            // warp w reads TMEM lanes 32*(w%4).., columns 32*(w/4)..; on the half
            // path the block of rows 32..63 (keys and queries) and columns 0..31
            // comes from the second product
            const int quad = warp & 3, chalf = warp >> 2, r = quad * 32 + lane;
            const uint32_t col = (path == 1 && (quad & 1) && chalf == 0) ? 64u : chalf * 32u;
            float v[32];
            if (ok) {
                tmem_ld32(tmem_addr(tmem, quad * 32, col), v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            wbar(bid);  // a1 is free: the MMAs consumed their operands
            if (r < C) {
                const int i = r;  // key-key row
                const float b = sm.beta[i];
#pragma unroll
                for (int jj = 0; jj < 32; jj += 4) {
                    const int j = chalf * 32 + jj;
                    float4 w;
                    w.x = (j < i && i < L) ? b * v[jj] : 0.f;
                    w.y = (j + 1 < i && i < L) ? b * v[jj + 1] : 0.f;
                    w.z = (j + 2 < i && i < L) ? b * v[jj + 2] : 0.f;
                    w.w = (j + 3 < i && i < L) ? b * v[jj + 3] : 0.f;
                    *reinterpret_cast<float4 *>(&R[i][j]) = w;
                }
            } else {
                const int i = r - C;  // query-key row
                float row[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = chalf * 32 + jj;
                    row[jj] = (j <= i && i < L) ? scale * v[jj] : 0.f;
                }
                store_quarter_f16_image(aqk, i, chalf * 4, row);
            }
        }
        if (hf == 0) gb[d] = exp2_approx(Gl);
        for (int idx = tid; idx < C * kRS / 4; idx += kPrepWorkerThreads)
            reinterpret_cast<float4 *>(&X[0][0])[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
        wbar(bid);

        // sec. 6.3: A^kk = (I + R)^-1, unit lower triangular, fp32.  The 16 x 16
        // diagonal blocks by right-looking substitution (one column per thread),
        // then the 32 x 32 diagonal blocks and the whole from block inverses:
        //   [A 0; B D]^-1 = [A^-1 0; -D^-1 B A^-1  D^-1]
        if (tid < C) {
            const int o = (tid >> 4) * 16, cc = tid & 15;
            float x[16], acc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                x[m] = m < cc ? 0.f : (m == cc ? 1.f : -acc[m]);
#pragma unroll
                for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(R[o + r][o + m], x[m], acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) X[o + r][o + cc] = x[r];
        }
        wbar(bid);
        solve_level16(R, X, Tb, tid, bid);
        solve_level32(R, X, Tb, tid, bid);
        // A^kk (rows i) and A^kk^T (rows j), f16
        if (tid < 2 * C) {
            const int row = tid >> 1, q4 = tid & 1;
            float v32[32], t32[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 xv = *reinterpret_cast<const float4 *>(&X[row][q4 * 32 + j]);
                v32[j] = xv.x;
                v32[j + 1] = xv.y;
                v32[j + 2] = xv.z;
                v32[j + 3] = xv.w;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) t32[j] = X[q4 * 32 + j][row];
            store_quarter_f16_image(b2, row, q4 * 4, v32);
            store_quarter_f16_image(akt, row, q4 * 4, t32);
        }
        fence_proxy_async();
        tc_fence_before();
        wbar(bid);
        // for the backward: A^kk and A^qk of this item out (read before Z is
        // staged over A^kk, below)
        if (bwd_aux && tid == 0) {
            bulk_s2g(bwd_aux + ch * kBwdAuxBytes, b2, 8192);
            bulk_s2g(bwd_aux + ch * kBwdAuxBytes + 8192, aqk, 8192);
            bulk_commit_group();
        }

        const int quad = warp & 3, chalf = warp >> 2;  // TMEM lanes 32*quad.., column half
        // W^T = (beta Gamma K)^T A^kk^T (TMEM cols 64..127) and Z = A^qk A^kk (cols
        // 0..63; rows 0..63 of a 128-row operand whose rows 64..127 are filler).
        if (tid == 0 && ok) {
            tc_fence_after();
            mma_panels(tmem + 64, smem_u32(a2), 0, smem_u32(b2), 0, 4, idesc_f16_f32(128, 64),
                       false);
            mma_panels(tmem, smem_u32(aqk), 0, smem_u32(akt), 0, 4, idesc_f16_f32(128, 64),
                       false);
            mma_commit(&sm.bar_mma);
        }
        if (ok) ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, wait_cycles);
        ok = __all_sync(0xffffffffu, ok);  // TMEM loads below are warp-collective
        mma_phase ^= 1u;
        tc_fence_after();
        if (bwd_aux) {
            // the copies of A^kk and A^qk have left shared memory
            if (tid == 0) bulk_wait_group_read<0>();
            wbar(bid);
        }
        {
            // thread = key channel d, token half chalf: W^T row d
            float v[32];
            if (ok) {
                tmem_ld32(tmem_addr(tmem, quad * 32, 64 + chalf * 32), v);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            store_quarter_f16_image(wt, d, chalf * 4, v);
            // Z rows 0..63 -> staging in the A^kk slot (read by the MMAs just done)
            if (quad < 2) {
                if (ok) tmem_ld32(tmem_addr(tmem, quad * 32, chalf * 32), v);
                store_quarter_f16_image(zst, quad * 32 + lane, chalf * 4, v);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        wbar(bid);

        // M' = K_end^T W (cols 0..127), P' = K_end^T A^kk (cols 128..191),
        // -Q'^T = -Q_hat^T + W^T A^qk^T (cols 192..255, onto what is there).
        if (tid == 0 && ok) {
            tc_fence_after();
            mma_panels(tmem, smem_u32(ket), 0, smem_u32(wt), 0, 4, idesc_f16_f32(128, 128),
                       false);
            mma_panels(tmem + 128, smem_u32(ket), 0, smem_u32(akt), 0, 4,
                       idesc_f16_f32(128, 64), false);
            mma_panels(tmem + 192, smem_u32(wt), 0, smem_u32(aqk), 0, 4, idesc_f16_f32(128, 64),
                       true);
            mma_commit(&sm.bar_mma);
        }
        if (ok) ok = mbar_wait_bounded(&sm.bar_mma, mma_phase, wait_cycles);
        ok = __all_sync(0xffffffffu, ok);  // TMEM loads below are warp-collective
        mma_phase ^= 1u;
        tc_fence_after();
        // Every operand is consumed: a1 becomes the staging of the image's first
        // 72 KB (-M' | P' | Q' keys 0..63 | . | Q' keys 64..127), Z waits in b1.
        if (ok) {
            float v0[32], v1[32];
            // -M' row d (key), columns (keys) 64*chalf.. -> image panel chalf
            tmem_ld32x2(tmem_addr(tmem, quad * 32, chalf * 64),
                        tmem_addr(tmem, quad * 32, chalf * 64 + 32), v0, v1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v0[j] = -v0[j];
                v1[j] = -v1[j];
            }
            store_quarter_f16_image(sm.a1 + IMG_MN + chalf * 16384, d, 0, v0);
            store_quarter_f16_image(sm.a1 + IMG_MN + chalf * 16384, d, 4, v1);
        }
        // -M' (with Z, staged before) starts out while P' and Q' are staged
        fence_proxy_async();
        wbar(bid);
        if (tid == 0) {
            bulk_s2g(img, sm.a1, IMG_P - IMG_MN);
            bulk_s2g(img + IMG_Z, zst, IMG_Q1 - IMG_Z);
            bulk_commit_group();
        }
        if (ok) {
            float v0[32];
            // P' row d, tokens 32*chalf..
            tmem_ld32(tmem_addr(tmem, quad * 32, 128 + chalf * 32), v0);
            store_quarter_f16_image(sm.a1 + IMG_P, d, chalf * 4, v0);
            // Q'[i][d] = s Gamma_i q_i[d] - (A^qk W)[i][d], tokens i = 32*chalf + jj,
            // as two 64-row panels
            tmem_ld32(tmem_addr(tmem, quad * 32, 192 + chalf * 32), v0);
            uint8_t *qs = sm.a1 + IMG_Q0 + (d >> 6) * 8192u;  // staged at IMG_Q0 and IMG_Z
#pragma unroll
            for (int jj = 0; jj < HALF; ++jj)
                *reinterpret_cast<__half *>(qs + sw128_offset(chalf * 32 + jj, d & 63)) =
                    __float2half_rn(-v0[jj]);
        }
        fence_proxy_async();
        tc_fence_before();
        wbar(bid);
        if (tid == 0) {
            // the rest of the image: [P' | Q' 0..63] in one piece, then Q' 64..127;
            // thread 0 waits for the stores (and publishes the image) after
            // issuing the next item's loads, or below after the last item
            bulk_s2g(img + IMG_P, sm.a1 + IMG_P, IMG_Z - IMG_P);
            bulk_s2g(img + IMG_Q1, sm.a1 + IMG_Z, IMG_GB - IMG_Q1);
            bulk_commit_group();
            sm.published = ch;
        }
        // one verdict per worker: after a wait that gave up, the worker stops
        if (wbar_or(bid, !ok)) {
            if (tid == 0) atomicExch(status, (int)KDA_ERR_TIMEOUT);
            break;
        }
    }
    if (tid == 0) {
        bulk_wait_group_all();  // the last image in global memory (the shared memory may go)
        if (flags && sm.published != ~0ull) {
            fence_proxy_async_global();
            flag_release(sc.ready + sm.published, 1u);
        }
        for (int i = 0; i < 3; ++i)
            if (sm.n_path[i]) atomicAdd(&g_path_counts[i], (unsigned long long)sm.n_path[i]);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(*tmem_slot, 256 * kPrepWorkers);
}

// ---------------------------------------------------------------------------
// 3. the inter-chunk scan: state only
// ---------------------------------------------------------------------------
// One CTA per (sequence, head, 64-wide value tile).  Per chunk n:
//   D2[n & 1]  = P' (beta V)            (issued one chunk ahead: no S_c in it)
//   D2[n & 1] += (-M') S_c              (the only dependency chain)
//   S_c+1      = Diag(Gamma_last) S_c + D2[n & 1]
// and the state entering each chunk goes out (f16, the output kernel's B
// operand image) for the fully parallel output pass.
constexpr int NSTAGE = 3;                   // image ring depth
constexpr int kScanPrefetch = 6;            // chunks ahead of the ring, into L2
constexpr uint32_t SCAN_IMG = IMG_P + 16384;  // -M' and P': the scan's part of an image
static_assert(SCAN_IMG == IMG_Q0, "the scan's operands lead the image");

struct ScanSmem {
    uint8_t st[NSTAGE][SCAN_IMG];  // -M' (32 KB) and P' (16 KB) of three chunks
    // B operands in MN-major (value columns contiguous) 128-byte-swizzled
    // layout: one row of 64 f16 values per K index
    uint8_t vs[NSTAGE][C * 128];   // the chunk's value tile, bf16 [64 tokens][64], 128 B swizzle
    uint8_t sb[2][D * 128];      // S_c:    K = 128 key rows (also the source of its
                                 // bulk copy out)
    uint8_t bv[2][C * 128];      // beta V: K = 64 token rows
    float gbs[NSTAGE][D + C];    // the chunk's Gamma_last [128] and beta [64]
    uint64_t full[NSTAGE];       // stage's -M' and P' loaded (bulk copy -> MMA issuer)
    uint64_t full_v[NSTAGE];     // stage's value tile, Gamma_last and beta loaded (-> compute)
    uint64_t empty[NSTAGE];      // stage consumed (tcgen05.commit -> producer)
    uint64_t ready_s;            // S_c operand written (compute -> issuer)
    uint64_t ready_bv[2];        // beta V operand written, per buffer
    uint64_t mma_s;              // chunk's state increment complete
    uint64_t ready_w[2];         // S_c operand written, for the writer of even / odd chunks
    uint32_t tmem;
    volatile int32_t copied[2];  // S_c images copied out of sb, per writer (writer -> compute)
    volatile int32_t issued;     // bulk copies issued (error path drains them)
    volatile int32_t abort_flag;
};

// warps 0-3 compute, 4 streams operands in, 5 issues MMAs, 6-7 write the S_c images out
constexpr int kScanThreads = 256;
constexpr uint32_t kScanTmemCols = 128;  // D2 ping-pong (2 x BV)
constexpr uint32_t kStateImg = D * 128;  // one value tile of S_c, f16 image

// Barrier over the 128 compute threads that also ORs a predicate over them,
// so that every one of them takes the same branch on the result.
__device__ __forceinline__ bool compute_barrier_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// 32 consecutive f16 values as 4 swizzled 16-byte chunks of one MN-major row.
__device__ __forceinline__ uint4 pack8_f16(const float *v) {
    uint4 u;
    u.x = pack_f16x2(v[0], v[1]);
    u.y = pack_f16x2(v[2], v[3]);
    u.z = pack_f16x2(v[4], v[5]);
    u.w = pack_f16x2(v[6], v[7]);
    return u;
}
__device__ __forceinline__ void store_row32_f16(uint8_t *img, uint32_t row, uint32_t chunk0,
                                                const float *v) {
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
        *reinterpret_cast<uint4 *>(img + sw128_chunk(row, chunk0 + c4)) = pack8_f16(v + c4 * 8);
}

// beta V of one token row, 32 value columns (64 bytes of bf16 in x), as f16
__device__ __forceinline__ void scale_row32(const uint4 (&x)[4], float b, float (&f)[32]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            f[i * 8 + 2 * y] = b * __uint_as_float(w[y] << 16);
            f[i * 8 + 2 * y + 1] = b * __uint_as_float(w[y] & 0xFFFF0000u);
        }
    }
}

__global__ void __launch_bounds__(kScanThreads, 1)
chunk_scan_kernel(const __grid_constant__ CUtensorMap v_map,
                  const float *__restrict__ initial_state,
                  const int32_t *__restrict__ cu, float *__restrict__ final_state, int32_t N,
                  int32_t T, int32_t H, Scratch sc, int32_t flags, int64_t sc_items,
                  long long wait_cycles, int *status) {
    extern __shared__ uint8_t smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // A programmatic dependent of the prep, which was launched before it and
    // whose CTAs are all running: the output pass may start setting up.  With
    // flags this kernel follows the prep item by item and never waits for its
    // grid; without, its producer waits for the whole prep below.  The chunk
    // table finished before the prep started, so its entries are read from L2.
    pdl_launch_dependents();
    const int32_t seq = blockIdx.x / NT, vt = blockIdx.x % NT, h = blockIdx.y;
    int32_t ta, tb;
    seq_bounds(cu, seq, T, ta, tb);
    const int32_t c_begin = __ldcg(sc.chunk_off + seq);
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
        if (tid == 0) {
            for (int i = 0; i < NSTAGE; ++i) {
                mbar_init(&sm.full[i], 1);
                mbar_init(&sm.full_v[i], 1);
                mbar_init(&sm.empty[i], 1);
            }
            mbar_init(&sm.ready_s, 128);
            mbar_init(&sm.ready_bv[0], 128);
            mbar_init(&sm.ready_bv[1], 128);
            mbar_init(&sm.mma_s, 1);
            mbar_init(&sm.ready_w[0], 128);
            mbar_init(&sm.ready_w[1], 128);
            sm.copied[0] = 0;
            sm.copied[1] = 0;
            sm.issued = 0;
            sm.abort_flag = 0;
            fence_mbar_init();
        }
        if (warp == 0) {
            tmem_alloc(&sm.tmem, kScanTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = sm.tmem;
        constexpr uint32_t IDESC = idesc_f16_f32(128, BV) | (1u << 16);  // B MN-major
        auto chunk_img = [&](int32_t n) {
            return sc.img + ((size_t)(c_begin + n) * H + h) * IMG_STRIDE;
        };
        auto state_img = [&](int32_t n) {
            return sc.sst + (((size_t)(c_begin + n) * H + h) * NT + vt) * kStateImg;
        };

        if (warp == 4) {
            // -------- producer: a chunk's value tile, Gamma_last and beta (on
            // full_v, for the compute warps) and its -M' and P' (on full, for
            // the MMAs), once its stage is free --------
            if (lane == 0) {
                if (!flags) pdl_wait_primaries();  // the prep has written every image
                for (int32_t n = 0; n < n_chunks; ++n) {
                    const int stg = n % NSTAGE;
                    // the image's flag first: its load latency then overlaps the
                    // wait for the stage
                    if (flags &&
                        !flag_wait_bounded(sc.ready + (size_t)(c_begin + n) * H + h,
                                           wait_cycles)) {
                        sm.abort_flag = 1;
                        break;
                    }
                    if (n >= NSTAGE) {
                        const bool got = mbar_wait_bounded(
                            &sm.empty[stg], (uint32_t)(n / NSTAGE - 1) & 1u, wait_cycles);
                        if (!got || sm.abort_flag) {
                            sm.abort_flag = 1;
                            break;
                        }
                    }
                    if (flags) fence_proxy_async_global();
                    // what the compute warps wait for (beta V of the chunk) ahead of
                    // the larger -M' and P' that only the MMAs read
                    mbar_arrive_expect_tx(&sm.full_v[stg],
                                          C * 128 + (D + C) * (uint32_t)sizeof(float));
                    bulk_g2s(sm.gbs[stg], chunk_img(n) + IMG_GB, (D + C) * sizeof(float),
                             &sm.full_v[stg]);
                    tma_load_3d(sm.vs[stg], &v_map, vt * BV, h, ta + n * C, &sm.full_v[stg]);
                    mbar_arrive_expect_tx(&sm.full[stg], SCAN_IMG);
                    bulk_g2s(sm.st[stg], chunk_img(n), SCAN_IMG, &sm.full[stg]);
                    sm.issued = n + 1;
                    // a few chunks further on into L2, so that their stage loads
                    // do not wait on HBM
                    if (n + kScanPrefetch < n_chunks) {
                        const uint8_t *im = chunk_img(n + kScanPrefetch);
                        bulk_prefetch_l2(im, SCAN_IMG);
                        bulk_prefetch_l2(im + IMG_GB, (D + C) * sizeof(float));
                        tma_prefetch_l2_3d(&v_map, vt * BV, h, ta + (n + kScanPrefetch) * C);
                    }
                }
            }
            __syncwarp();
        } else if (warp == 5) {
            // -------- MMA issuer --------
            if (lane == 0) {
                int32_t done = 0;  // chunks whose state group was issued
                for (int32_t n = 0; n < n_chunks; ++n) {
                    const int stg = n % NSTAGE;
                    const uint8_t *img = sm.st[stg];
                    const uint32_t d2 = tmem + (uint32_t)(n & 1) * BV;
                    // P' (beta V): needs only the chunk's own operands
                    bool got = mbar_wait_bounded(&sm.full[stg], (uint32_t)(n / NSTAGE) & 1u,
                                                 wait_cycles) &&
                               mbar_wait_bounded(&sm.ready_bv[n & 1], (uint32_t)(n >> 1) & 1u,
                                                 wait_cycles);
                    if (!got || sm.abort_flag) {
                        sm.abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                    mma_kmajor_a_mn_b(d2, smem_u32(img + IMG_P), 0, smem_u32(sm.bv[n & 1]), 4,
                                      IDESC, false);
                    // (-M') S_c once the state is in
                    got = mbar_wait_bounded(&sm.ready_s, (uint32_t)n & 1u, wait_cycles);
                    if (!got || sm.abort_flag) {
                        sm.abort_flag = 1;
                        mma_commit(&sm.empty[stg]);  // keeps the drain below exact
                        done = n + 1;
                        break;
                    }
                    tc_fence_after();
                    mma_kmajor_a_mn_b(d2, smem_u32(img + IMG_MN), 16384,
                                      smem_u32(sm.sb[n & 1]), 8, IDESC, true);
                    mma_commit(&sm.mma_s);
                    mma_commit(&sm.empty[stg]);  // the stage may be refilled after these
                    done = n + 1;
                }
                // the stage-release arrivals of the last chunks (no one else waits
                // for them) land before the shared memory goes away; the last one
                // also means every MMA issued is done
                for (int32_t j = max(done - NSTAGE, 0); j < done; ++j)
                    if (!mbar_wait_bounded(&sm.empty[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u,
                                           wait_cycles))
                        sm.abort_flag = 1;
            }
            __syncwarp();
        } else if (warp >= 6) {
            // -------- state writers: the S_c images out (with flags: and their
            // flags, for the output pass), off the compute warps' chain.  Two
            // of them take the chunks in turn, so that each waits for its copy
            // to land and publishes it with no other copy of its own in flight
            // (a release waits for those) while the other copies the next.
            const int b = warp - 6;
            if (lane == 0) {
                for (int32_t n = b; n < n_chunks; n += 2) {
                    // S_c in sb[n & 1], written and fenced by the compute warps
                    if (!mbar_wait_bounded(&sm.ready_w[b], (uint32_t)(n >> 1) & 1u,
                                           wait_cycles) ||
                        sm.abort_flag) {
                        sm.abort_flag = 1;
                        break;
                    }
                    bulk_s2g(state_img(n), sm.sb[n & 1], kStateImg);
                    bulk_commit_group();
                    bulk_wait_group_read<0>();
                    sm.copied[b] = (n >> 1) + 1;
                    if (flags) {
                        bulk_wait_group_all();
                        fence_proxy_async_global();
                        flag_release(sc.ready + (size_t)sc_items +
                                         ((size_t)(c_begin + n) * H + h) * NT + vt,
                                     1u);
                    }
                }
                bulk_wait_group_all();  // state images written
            }
            __syncwarp();
        } else {
            // ---------------- compute warps ----------------
            // Everything a chunk needs arrives with its stage (no global loads in
            // the loop: a barrier would wait for them).  beta V: thread -> token
            // row tid/2, 32 value columns.
            const int vi = tid >> 1, vh = tid & 1;
            auto build_bv = [&](int32_t n) {
                const int stg = n % NSTAGE;
                const bool valid = vi < tb - (ta + n * C);  // rows past the sequence are zero
                const float b = valid ? sm.gbs[stg][D + vi] : 0.f;
                uint4 x[4];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    x[c4] = *reinterpret_cast<const uint4 *>(sm.vs[stg] +
                                                             sw128_chunk(vi, vh * 4 + c4));
                float f[32];
                scale_row32(x, b, f);
                store_row32_f16(sm.bv[n & 1], vi, vh * 4, f);
                fence_proxy_async();
                mbar_arrive(&sm.ready_bv[n & 1]);
            };
            auto wait_full = [&](int32_t n) {
                if (!mbar_wait_bounded(&sm.full_v[n % NSTAGE], (uint32_t)(n / NSTAGE) & 1u,
                                       wait_cycles))
                    sm.abort_flag = 1;
            };
            // S_c of chunk n as the MMA's B operand (f16); the same image goes out
            // to global memory for the output pass (the writer warp copies it)
            auto put_state = [&](int32_t n) {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8)
                    *reinterpret_cast<uint4 *>(sm.sb[n & 1] + sw128_chunk(tid, c8)) =
                        pack8_f16(&S[c8 * 8]);
                fence_proxy_async();
            };

            wait_full(0);
            float g = sm.gbs[0][tid];  // Gamma_last of chunk n (read before its stage is freed)
            build_bv(0);
            put_state(0);
            for (int32_t n = 0; n < n_chunks; ++n) {
                if (compute_barrier_or(sm.abort_flag != 0)) break;
                tc_fence_before();
                mbar_arrive(&sm.ready_s);
                mbar_arrive(&sm.ready_w[n & 1]);
                const bool more = n + 1 < n_chunks;
                float g_next = 0.f;
                if (more) {
                    // beta V of the next chunk (its buffer was last read two chunks ago)
                    wait_full(n + 1);
                    g_next = sm.gbs[(n + 1) % NSTAGE][tid];
                    build_bv(n + 1);
                }
                if (!mbar_wait_bounded(&sm.mma_s, (uint32_t)n & 1u, wait_cycles))
                    sm.abort_flag = 1;
                tc_fence_after();
                {
                    const uint32_t d2 = tmem + (uint32_t)(n & 1) * BV;
                    float ds0[32], ds1[32];
                    tmem_ld32x2(tmem_addr(d2, warp * 32, 0), tmem_addr(d2, warp * 32, 32), ds0,
                                ds1);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        S[j] = fmaf(g, S[j], ds0[j]);
                        S[32 + j] = fmaf(g, S[32 + j], ds1[j]);
                    }
                }
                g = g_next;
                if (more) {
                    // sb[(n + 1) & 1] holds S_n-1: wait until its writer has copied
                    // it out (issued a chunk ago: normally long done)
                    if (n >= 1) {
                        const int wb = (n - 1) & 1;
                        const int32_t need = ((n - 1) >> 1) + 1;
                        if (sm.copied[wb] < need) {
                            const long long t0 = clock64();
                            while (sm.copied[wb] < need) {
                                if (clock64() - t0 > wait_cycles) {
                                    sm.abort_flag = 1;
                                    break;
                                }
                            }
                        }
                    }
                    put_state(n + 1);
                }
            }
        }
        __syncthreads();
        if (sm.abort_flag) {
            ok = false;
            if (tid == 0) {
                atomicExch(status, (int)KDA_ERR_TIMEOUT);
                // copies already in flight land before the shared memory goes away
                const int32_t iss = sm.issued;
                for (int32_t j = max(iss - NSTAGE, 0); j < iss; ++j) {
                    (void)mbar_wait_bounded(&sm.full_v[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u,
                                            wait_cycles);
                    (void)mbar_wait_bounded(&sm.full[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u,
                                            wait_cycles);
                }
            }
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

// ---------------------------------------------------------------------------
// 4. outputs: O = Q' S_c + Z (beta V), one CTA per (chunk, head)
// ---------------------------------------------------------------------------
// Fully parallel once the scan has written every S_c.  128 threads; the
// A operands are 128-row tiles whose first 64 rows are filler (see IMG_*),
// so the outputs sit in TMEM lanes 64..127 (warps 2 and 3).
// The output pass's A operands: [filler ; Q' keys 0..63], [Z ; Q' keys 64..127]
// and [Q' keys 0..63 ; Z] -- 128-row panels whose upper 64 rows only produce
// TMEM lanes that are never read.  The first 8 KB (filler) is cleared in
// shared memory, the other 24 KB come from the image.
constexpr uint32_t OUT_IMG_OFF = IMG_Q0 - 8192;
constexpr uint32_t OUT_IMG_BYTES = IMG_GB - OUT_IMG_OFF;
constexpr uint32_t OUT_FILL = 8192;
static_assert(OUT_IMG_OFF % 1024 == 0 && OUT_IMG_BYTES == 32768, "output operand region");

struct OutSmem {
    uint8_t qz[OUT_IMG_BYTES];   // [filler ; Q'] panels and [filler ; Z]
    uint8_t sS[NT][kStateImg];   // S_c, one MN-major image per value tile
    uint8_t bv[NT][C * 128];     // beta V, per value tile
    uint8_t vin[NT][C * 128];    // the chunk's value tiles (TMA, 128-byte swizzle)
    float beta[C];
    uint64_t bar_in, bar_mma;
    uint32_t tmem;
};
constexpr int kOutThreads = 128;

template <typename TOut>
__global__ void __launch_bounds__(kOutThreads)
chunk_out_kernel(const __grid_constant__ CUtensorMap out_map, const __grid_constant__ CUtensorMap v_map,
                 const int32_t *__restrict__ cu, TOut *__restrict__ out, int32_t N, int32_t T,
                 int32_t H, Scratch sc, int32_t flags, int64_t sc_items,
                 long long wait_cycles, int *status) {
    extern __shared__ uint8_t smem_raw[];
    OutSmem &sm = *reinterpret_cast<OutSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    // heads fastest: the order in which the scan finishes the chunks' states
    const int32_t c = (int32_t)(blockIdx.x / (unsigned)H), h = (int32_t)(blockIdx.x % (unsigned)H);
    const int2 tok = __ldcg(sc.chunk_tok + c);  // the chunk table finished long before
    const int32_t t0 = tok.x, L = tok.y;
    if (L <= 0) return;
    const uint8_t *img = sc.img + ((size_t)c * H + h) * IMG_STRIDE;

    // Without flags: the scan (and before it the prep) has finished.  With
    // flags (running beside the prep's last workers and the scan, both
    // launched before this kernel and running): this chunk's image and both
    // value tiles of its S_c are up.  A wait that runs out leaves the status
    // set and garbage outputs, never a hang.
    if (!flags) pdl_wait_primaries();
    if (tid == 0) {
        if (flags) {
            bool got = flag_wait_bounded(sc.ready + (size_t)c * H + h, wait_cycles);
            for (int t = 0; t < NT && got; ++t)
                got = flag_wait_bounded(sc.ready + sc_items + ((size_t)c * H + h) * NT + t,
                                        wait_cycles);
            if (!got) atomicExch(status, (int)KDA_ERR_TIMEOUT);
            fence_proxy_async_global();
        }
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
        // Q'/Z, both S_c tiles, both value tiles and beta, all on one barrier
        mbar_arrive_expect_tx(&sm.bar_in, OUT_IMG_BYTES - OUT_FILL + NT * kStateImg +
                                              NT * C * 128 + C * (uint32_t)sizeof(float));
        bulk_g2s(sm.qz + OUT_FILL, img + OUT_IMG_OFF + OUT_FILL, OUT_IMG_BYTES - OUT_FILL,
                 &sm.bar_in);
        bulk_g2s(sm.sS, sc.sst + ((size_t)c * H + h) * NT * kStateImg, NT * kStateImg,
                 &sm.bar_in);
#pragma unroll
        for (int t = 0; t < NT; ++t) tma_load_3d(sm.vin[t], &v_map, t * BV, h, t0, &sm.bar_in);
        bulk_g2s(sm.beta, img + IMG_GB + D * sizeof(float), C * sizeof(float), &sm.bar_in);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 128);
        tmem_relinquish();
    }
    // the filler rows (made visible to the MMAs by the proxy fence below)
    for (int i = tid; i < (int)(OUT_FILL / 16); i += 128)
        reinterpret_cast<uint4 *>(sm.qz)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    bool ok = mbar_wait_bounded(&sm.bar_in, 0, wait_cycles);
    // beta V: thread -> token tid / 2, value tile tid % 2 (rows past the
    // sequence, another sequence's tokens or zeros past T, get beta 0)
    {
        const int i = tid >> 1, half = tid & 1;
        const float b = i < L ? sm.beta[i] : 0.f;
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
            uint4 x[4];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                x[c4] = *reinterpret_cast<const uint4 *>(sm.vin[half] +
                                                         sw128_chunk(i, q4 * 4 + c4));
            float f[32];
            scale_row32(x, b, f);
            store_row32_f16(sm.bv[half], i, q4 * 4, f);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        constexpr uint32_t IDESC = idesc_f16_f32(128, BV) | (1u << 16);  // B MN-major
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint32_t d = tmem + t * BV;
            mma_kmajor_a_mn_b(d, smem_u32(sm.qz), 16384, smem_u32(sm.sS[t]), 8, IDESC, false);
            mma_kmajor_a_mn_b(d, smem_u32(sm.qz) + (IMG_Z - 8192 - OUT_IMG_OFF), 0,
                              smem_u32(sm.bv[t]), 4, IDESC, true);
        }
        mma_commit(&sm.bar_mma);
    }
    if (ok) ok = mbar_wait_bounded(&sm.bar_mma, 0, wait_cycles);
    tc_fence_after();
    ok = !__syncthreads_or(!ok);  // one verdict for all (warps 2-3 share a barrier below)
    if (ok && warp >= 2) {
        const int i = tid - 64;  // token
        if (L == C) {
            // swizzled 128-byte column panels (over the consumed operands), then
            // TMA tensor stores
            uint8_t *ob = sm.qz;
            static_assert(C * D * 4 <= OUT_IMG_BYTES + NT * kStateImg, "staging fits");
            constexpr int kPanelCols = 128 / (int)sizeof(TOut);
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                float o[32];
                tmem_ld32(tmem_addr(tmem, warp * 32, cb), o);
#pragma unroll
                for (int j = 0; j < 32; j += 16 / (int)sizeof(TOut)) {
                    const int col = cb + j, pnl = col / kPanelCols;
                    const int chunk = (col % kPanelCols) * (int)sizeof(TOut) / 16;
                    uint4 u;
                    if constexpr (sizeof(TOut) == 2) {
                        u.x = pack_bf16x2(o[j], o[j + 1]);
                        u.y = pack_bf16x2(o[j + 2], o[j + 3]);
                        u.z = pack_bf16x2(o[j + 4], o[j + 5]);
                        u.w = pack_bf16x2(o[j + 6], o[j + 7]);
                    } else {
                        u = make_uint4(__float_as_uint(o[j]), __float_as_uint(o[j + 1]),
                                       __float_as_uint(o[j + 2]), __float_as_uint(o[j + 3]));
                    }
                    *reinterpret_cast<uint4 *>(ob + pnl * (C * 128) + sw128_chunk(i, chunk)) = u;
                }
            }
            fence_proxy_async();
            asm volatile("bar.sync 2, 64;" ::: "memory");
            if (tid == 64) {
#pragma unroll
                for (int pnl = 0; pnl < D / kPanelCols; ++pnl)
                    tma_store_3d(&out_map, ob + pnl * (C * 128), pnl * kPanelCols, h, t0);
                bulk_commit_group();
                bulk_wait_group_read<0>();
            }
        } else {
            // a sequence's last, partial chunk: valid rows only, plain stores
            // (the TMEM loads are warp-collective: every lane takes part)
            TOut *dst = out + ((size_t)(t0 + min(i, L - 1)) * H + h) * D;
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
                float o[32];
                tmem_ld32(tmem_addr(tmem, warp * 32, cb), o);
                if (i >= L) continue;
                if constexpr (sizeof(TOut) == 2) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 u;
                        u.x = pack_bf16x2(o[j], o[j + 1]);
                        u.y = pack_bf16x2(o[j + 2], o[j + 3]);
                        u.z = pack_bf16x2(o[j + 4], o[j + 5]);
                        u.w = pack_bf16x2(o[j + 6], o[j + 7]);
                        *reinterpret_cast<uint4 *>(dst + cb + j) = u;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(dst + cb + j) =
                            make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
                }
            }
        }
    }
    if (!ok && tid == 0) atomicExch(status, (int)KDA_ERR_TIMEOUT);
    if (!ok && tid == 0) {
        // let the loads land before the shared memory goes away
        (void)mbar_wait_bounded(&sm.bar_in, 0, wait_cycles);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

constexpr size_t kPrepSmem = kPrepWorkers * kPrepWorkerBytes + 16 + 1024;
constexpr size_t kScanSmem = sizeof(ScanSmem) + 1024;
constexpr size_t kOutSmem = sizeof(OutSmem) + 1024;
static_assert(kScanSmem <= 227 * 1024, "scan shared memory");
static_assert(2 * kOutSmem <= 228 * 1024 - 2 * 1024, "two output CTAs per SM");
static_assert(kPrepSmem <= 227 * 1024, "prep shared memory (two workers)");
static_assert(kPrepSmem > 114 * 1024, "one prep CTA per SM: the SMs it leaves take the scan");
// Largest prep run beside the scan on the SMs the scan leaves; longer ones
// take every SM first, and the scan follows (the tail order).
constexpr size_t kStreamMaxItems = 1u << 16;
// Bounded waits give up after this many SM clocks (~1 s at 2 GHz).
constexpr long long kWaitCycles = 2000000000LL;

}  // namespace

size_t chunk_tc_workspace_bytes(int32_t N, int32_t T, int32_t H) {
    const size_t nch = max_chunks(N, T) * (size_t)H;
    return align256(nch * IMG_STRIDE) + align256(nch * NT * (size_t)(D * 128)) +
           align256(nch * (1 + NT) * sizeof(uint32_t)) + align256(max_chunks(N, T) * sizeof(int2)) +
           align256(((size_t)N + 1) * sizeof(int32_t));
}

ChunkScratchView chunk_tc_scratch_view(void *workspace, int32_t N, int32_t T, int32_t H) {
    static_assert(IMG_STRIDE == kChunkImgStride && NT == 2 && kStateImg == 16384,
                  "the layout the backward reads");
    const Scratch sc = carve(workspace, N, T, H);
    ChunkScratchView v;
    v.img = sc.img;
    v.sst = sc.sst;
    v.chunk_tok = sc.chunk_tok;
    v.chunk_off = sc.chunk_off;
    v.max_chunks = max_chunks(N, T);
    return v;
}

cudaError_t chunk_path_counts(uint64_t counts[3], bool clear) {
    unsigned long long v[3] = {0, 0, 0};
    cudaError_t e = cudaMemcpyFromSymbol(v, g_path_counts, sizeof(v));
    if (e == cudaSuccess && clear) {
        const unsigned long long z[3] = {0, 0, 0};
        e = cudaMemcpyToSymbol(g_path_counts, z, sizeof(z));
    }
    for (int i = 0; i < 3; ++i) counts[i] = (uint64_t)v[i];
    return e;
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
                     int32_t T, int32_t H, uint32_t box_x, CUtensorMapSwizzle swz) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
    const cuuint32_t box[3] = {box_x, 1u, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// KDA_LAUNCH_ORDER=sequential runs every call in the sequential order (for
// profilers that time one kernel at a time with the whole GPU to itself).
bool sequential_order_forced() {
    static const bool forced = [] {
        const char *order = std::getenv("KDA_LAUNCH_ORDER");
        return order && std::strcmp(order, "sequential") == 0;
    }();
    return forced;
}

cudaError_t launch_chunk_tc(const ChunkArgs &a, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
    if (workspace_bytes < chunk_tc_workspace_bytes(a.N, a.T, a.H) || !workspace)
        return cudaErrorInvalidValue;
    const Scratch sc = carve(workspace, a.N, a.T, a.H);
    // Four launches: table -> prep -> scan -> output, each after the table a
    // programmatic dependent of the kernel before it (its CTAs may become
    // resident while that kernel still runs).  No kernel ever waits on work
    // of a kernel launched after it, so any schedule the GPU picks -- one
    // kernel at a time included -- completes.
    //
    // Overlapped order (the scan's CTAs fit in half of the SMs): the prep is
    // persistent and triggers its dependents as soon as its CTAs run; with up
    // to kStreamMaxItems items it takes only the SMs that the scan's CTAs
    // leave, so the scan runs beside it, following each image through its
    // flag; with more, it takes every SM and the scan starts on the SMs its
    // workers leave when the items run out (the tail order).  The output
    // kernel follows the images and the scan's states through flags, on SMs
    // that prep workers leave.  The waits are on CTAs already running.
    //
    // Sequential order (more scan CTAs than half of the SMs, per-kernel
    // events requested, or KDA_LAUNCH_ORDER=sequential): each kernel waits on
    // griddepcontrol for the whole kernel ahead before it reads its results.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    const bool timed = a.clock && a.clock->max_events > 0;
    const bool diag = a.diag_withhold_prep != 0;
    const size_t n_items = max_chunks(a.N, a.T) * (size_t)a.H;  // prep items
    const size_t scan_ctas = (size_t)a.N * NT * (size_t)a.H;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    // the kernels hand work over through flags (overlapped order)
    const bool flags = diag || (!timed && !sequential_order_forced() && a.T > 0 && sms > 0 &&
                                2 * scan_ctas <= (size_t)sms);
    const bool beside = flags && n_items <= kStreamMaxItems;
    size_t prep_ctas = sms > 0 ? (size_t)sms : 1;
    if (beside) prep_ctas = std::max<size_t>(1, (size_t)sms - scan_ctas);
    prep_ctas = std::max<size_t>(
        1, std::min(prep_ctas, (n_items + kPrepWorkers - 1) / (size_t)kPrepWorkers));
    const long long wait_cycles = a.wait_cycles > 0 ? a.wait_cycles : kWaitCycles;
    auto config = [&](dim3 grid, int threads, size_t smem, bool dependent) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = pdl;
        cfg.numAttrs = (dependent && !timed) ? 1u : 0u;
        return cfg;
    };
    // Every kernel is set up (and so loaded, under lazy module loading) before
    // the first launch, and every tensor map encoded, so that the launches
    // follow one another without host work in between.
    auto prep = a.pro ? chunk_prep_kernel<true> : chunk_prep_kernel<false>;
    auto out_kernel_f32 = chunk_out_kernel<float>;
    auto out_kernel_bf16 = chunk_out_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPrepSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kScanSmem);
    if (e == cudaSuccess)
        e = a.out_f32 ? cudaFuncSetAttribute(out_kernel_f32,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kOutSmem)
                      : cudaFuncSetAttribute(out_kernel_bf16,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kOutSmem);
    if (e != cudaSuccess) return e;

    PrepMaps maps;
    CUtensorMap v_map, out_map;
    memset(&maps, 0, sizeof(maps));
    memset(&v_map, 0, sizeof(v_map));
    memset(&out_map, 0, sizeof(out_map));
    if (a.T > 0) {
        if (!encode_tile_map(&maps.q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H / a.G) ||
            !encode_tile_map(&maps.k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H / a.G) ||
            !encode_tile_map(&maps.g, a.log_alpha, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H))
            return cudaErrorInvalidValue;
        // value tiles [64 tokens x 64 columns] of one head, 128-byte swizzle
        if (!encode_tile_map(&v_map, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H, BV,
                             CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (a.T > 0 && !a.skip_out) {
        // output tiles [64 tokens x 128-byte column panel] of one head
        auto enc = tensor_map_encoder();
        const size_t es = a.out_f32 ? 4 : 2;
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.H, (cuuint64_t)a.T};
        const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)a.H * D * es};
        const cuuint32_t box[3] = {(cuuint32_t)(128 / es), 1u, (cuuint32_t)C};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        if (!enc ||
            enc(&out_map, a.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                3, a.out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    const size_t n_ready = flags ? n_items * (1 + NT) : 0;  // image and state flags
    const unsigned table_ctas = 1u + (unsigned)std::min<size_t>(n_ready / 16384, 63);
    chunk_table_kernel<<<table_ctas, 1024, 0, stream>>>(a.cu_seqlens, a.N, a.T, sc.chunk_off,
                                                        sc.chunk_tok, sc.ready, n_ready);
    a.clock->mark(stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // The diagnostic run withholds the prep: the scan's first flag is never
    // published and its bounded waits run out.
    const bool run_prep = a.T > 0 && !diag;
    if (run_prep) {
        const cudaLaunchConfig_t cfg =
            config(dim3((unsigned)prep_ctas), kPrepThreads, kPrepSmem, true);
        e = cudaLaunchKernelEx(&cfg, prep, maps, static_cast<const __nv_bfloat16 *>(a.q),
                               static_cast<const __nv_bfloat16 *>(a.k), a.beta, a.scale, a.H,
                               a.G, a.pro, a.gbias, a.galog, sc, (uint32_t)n_items,
                               (int32_t)flags, wait_cycles, a.status, a.bwd_aux);
        if (e != cudaSuccess) return e;
    }
    a.clock->mark(stream);

    {
        // a plain launch when no prep runs ahead of it (it reads the table)
        const cudaLaunchConfig_t cfg = config(dim3((unsigned)(a.N * NT), (unsigned)a.H),
                                              kScanThreads, kScanSmem, run_prep);
        e = cudaLaunchKernelEx(&cfg, chunk_scan_kernel, v_map, a.initial_state,
                               static_cast<const int32_t *>(a.cu_seqlens), a.final_state, a.N,
                               a.T, a.H, sc, (int32_t)flags, (int64_t)n_items, wait_cycles,
                               a.status);
        if (e != cudaSuccess) return e;
    }
    a.clock->mark(stream);

    if (run_prep && !a.skip_out) {
        const cudaLaunchConfig_t cfg = config(dim3((unsigned)n_items), kOutThreads, kOutSmem, true);
        const int32_t *cu = static_cast<const int32_t *>(a.cu_seqlens);
        if (a.out_f32) {
            e = cudaLaunchKernelEx(&cfg, out_kernel_f32, out_map, v_map, cu,
                                   static_cast<float *>(a.out), a.N, a.T, a.H, sc,
                                   (int32_t)flags, (int64_t)n_items, wait_cycles, a.status);
        } else {
            e = cudaLaunchKernelEx(&cfg, out_kernel_bf16, out_map, v_map, cu,
                                   static_cast<__nv_bfloat16 *>(a.out), a.N, a.T, a.H, sc,
                                   (int32_t)flags, (int64_t)n_items, wait_cycles, a.status);
        }
        if (e != cudaSuccess) return e;
    }
    a.clock->mark(stream);
    return cudaGetLastError();
}

}  // namespace kda
