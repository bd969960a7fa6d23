// kda_backward_chunk.cu -- the chunkwise backward (training).
//
// The pages derive no gradients ("Kimi Unveils Delta Attention and K3
// Architecture Updates", sec. 6: the chunkwise form serves training).  The
// chunk form of sec. 6 differentiated by reverse mode has one serial part,
// the forward scan transposed on the same folded factors:
//
//   dS_c = Diag(exp(G_last)) dS_{c+1} - M'^T dS_{c+1} + Q'^T dO_c
//
// and, once S_c and dS_{c+1} are known at every chunk boundary, each chunk's
// gradients are independent of the others.  This form:
//   1. runs the forward engine without its output pass; its workspace keeps
//      every chunk's f16 M', Q', exp(G_last) and the f16 state S_c entering
//      the chunk, and its prep also stores every chunk's A^kk and A^qk;
//   2. chunk_bwd_aux_kernel: -M'^T as a bf16 operand image and
//      X_c = Q'^T dO_c (one tcgen05 kind::tf32 product) per (chunk, head);
//   3. chunk_rscan_kernel: the reverse scan, one kind::f16 product on bf16
//      operands per chunk on the chain, writing dS_{c+1} at every boundary
//      (as the gradient pass's transposed tf32 operand tiles and as
//      value-contiguous fp32 panels) and dS at every sequence start (the
//      initial-state gradient);
//   4. the per-chunk gradient pass on the tensor cores (kda_backward_grad.cu).
// Every product that carries a gradient keeps fp32 range (tf32 or bf16
// operands): f16 operands lose gradients of training size to underflow.  The
// reverse scan's state operand is bf16 (its fp32 state stays in registers):
// the rounding of that one product's operands moves the gradients by far less
// than the gradient pass's own tf32 roundings.
#include <algorithm>
#include <cstdint>
#include <cstring>

#include <cuda_bf16.h>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {
using namespace tc;


constexpr int AD = 128, AC = 64;
constexpr uint32_t A_IMG_STRIDE = 74752, A_IMG_MN = 0, A_IMG_Q0 = 49152, A_IMG_Q1 = 65536,
                   A_IMG_GB = 73728;
constexpr long long kAWait = 2000000000LL;

struct AuxSmem {
    uint8_t mt[2 * 16384];   // -M'^T staging (bf16), then the bulk copy out
    uint8_t qt[2 * 16384];   // A: Q'^T, 128 rows x 64 tokens, 2 panels
    uint8_t dt[2 * 16384];   // B: dO^T, 128 rows (d_v) x 64 tokens, 2 panels
    uint8_t mn[2 * 16384];   // -M' f16 panels (bulk copy in)
    uint8_t q0[8192], q1[8192];  // Q' f16 panels (keys 0..63, 64..127)
    uint8_t dtile[AC * AD * 2];  // the dO tile, bf16 [64 tokens][128]
    float gl[2][AD];             // exp(G_last), by item parity (in while the last goes out)
    uint64_t bar_in, bar_mma;
    uint32_t tmem;
};
constexpr size_t kAuxSmem = sizeof(AuxSmem) + 1024;
static_assert(kAuxSmem <= 227 * 1024, "aux shared memory");

__device__ __forceinline__ float f16_at(const uint8_t *panel, uint32_t row, uint32_t col) {
    return __half2float(*reinterpret_cast<const __half *>(panel + sw128_offset(row, col)));
}

// dO as TMA tiles of one head's [64 tokens x 128 channels] (bf16)
struct AuxMaps {
    CUtensorMap d;
};

// Persistent: CTA b takes items b, b + grid, ... in the order the reverse
// scan consumes them (chunks from the last, heads fastest).  With flags,
// each item's outputs are published once they are in global memory (thread
// 0 waits for its bulk stores and releases the item's flag after issuing the
// next item's loads), so the reverse scan, launched as a programmatic
// dependent once every CTA of this grid runs, follows item by item.
__global__ void __launch_bounds__(256, 1)
chunk_bwd_aux_kernel(const __grid_constant__ AuxMaps maps, const uint8_t *__restrict__ img_base,
                     const int2 *__restrict__ chunk_tok, int32_t has_d_out,
                     uint8_t *__restrict__ mt_img, float *__restrict__ x_tiles,
                     float *__restrict__ glv, int32_t H, int32_t max_chunks,
                     uint32_t *__restrict__ ready, int *status) {
    extern __shared__ uint8_t smem_raw[];
    AuxSmem &sm = *reinterpret_cast<AuxSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    // the reverse scan may start: it waits on items of this running grid
    pdl_launch_dependents();
    uint8_t *dtile = sm.dtile;
    if (tid == 0) {
        mbar_init(&sm.bar_in, 1);
        mbar_init(&sm.bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    const size_t n_items = (size_t)max_chunks * H;
    // this CTA's items in order, skipping chunks that do not exist
    auto chunk_of = [&](size_t k) { return max_chunks - 1 - (int32_t)(k / (size_t)H); };
    auto next_valid = [&](size_t k) {
        while (k < n_items && chunk_tok[chunk_of(k)].y <= 0) k += gridDim.x;
        return k;
    };
    // one item's inputs: -M', Q', exp(G_last) (into the parity's slot) and dO
    auto issue = [&](size_t k, uint32_t par) {
        const int32_t c = chunk_of(k), h = (int32_t)(k % (size_t)H);
        const uint8_t *img = img_base + ((size_t)c * H + h) * A_IMG_STRIDE;
        mbar_arrive_expect_tx(&sm.bar_in,
                              2 * 16384 + 2 * 8192 + AD * 4 + (has_d_out ? AC * AD * 2 : 0));
        bulk_g2s(sm.mn, img + A_IMG_MN, 2 * 16384, &sm.bar_in);
        bulk_g2s(sm.q0, img + A_IMG_Q0, 8192, &sm.bar_in);
        bulk_g2s(sm.q1, img + A_IMG_Q1, 8192, &sm.bar_in);
        bulk_g2s(sm.gl[par], img + A_IMG_GB, AD * 4, &sm.bar_in);
        if (has_d_out) tma_load_3d(dtile, &maps.d, 0, h, chunk_tok[c].x, &sm.bar_in);
    };
    size_t published = ~size_t(0);  // thread 0: the item whose flag is still to go up
    uint32_t phase = 0;
    bool ok = true;
    size_t k = next_valid(blockIdx.x);
    if (tid == 0 && k < n_items) issue(k, 0);
    while (k < n_items) {
        const int32_t c = chunk_of(k), h = (int32_t)(k % (size_t)H);
        const int32_t L = chunk_tok[c].y;
        const size_t item = (size_t)c * H + h;
        const size_t k_next = next_valid(k + gridDim.x);
        ok = mbar_wait_bounded(&sm.bar_in, phase, kAWait) && ok;
        // dO^T (B operand): element (n, i) = dO[t0 + i][h][n], rows i >= L zero.
        // Thread -> column n = tid % 128, tokens i = tid / 128, +2, ...
        {
            const int n = tid & 127;
            const unsigned short *tile = reinterpret_cast<const unsigned short *>(dtile);
#pragma unroll 8
            for (int i = tid >> 7; i < AC; i += 2) {
                const float x = (has_d_out && i < L)
                                    ? __uint_as_float((uint32_t)tile[i * AD + n] << 16)
                                    : 0.f;
                *reinterpret_cast<float *>(sm.dt + (i >> 5) * 16384u +
                                           sw128_offset_f32(n, i & 31)) = x;
            }
        }
        if (ok) {
            if (tid < 128) {
                // -M'^T row i = column i of -M': (-M')[j][i] at panel i/64, row j;
                // bf16 (the reverse scan's product is kind::f16 on bf16 operands:
                // the gradient keeps fp32 range)
                const int i = tid;
                const uint8_t *src = sm.mn + (i >> 6) * 16384u;
#pragma unroll 2
                for (int p = 0; p < 2; ++p) {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const int j = p * 64 + c8 * 8;
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                f16_at(src, j + 2 * e, i & 63), f16_at(src, j + 2 * e + 1, i & 63));
                            w[e] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(sm.mt + p * 16384u + sw128_chunk(i, c8)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            } else {
                // Q'^T row d = column d of Q': Q'[i][d] at the panel of d, row i
                const int d = tid - 128;
                const uint8_t *src = d < 64 ? sm.q0 : sm.q1;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const int i = p * 32 + c4 * 4;
                        float4 v;
                        v.x = f16_at(src, i, d & 63);
                        v.y = f16_at(src, i + 1, d & 63);
                        v.z = f16_at(src, i + 2, d & 63);
                        v.w = f16_at(src, i + 3, d & 63);
                        *reinterpret_cast<float4 *>(sm.qt + p * 16384u + sw128_chunk(d, c4)) = v;
                    }
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();  // -M', Q' and the dO tile are read: the next item's may land
        if (tid == 0) {
            if (ok && k_next < n_items) issue(k_next, phase ^ 1u);
            // the previous item's outputs are in global memory: publish it
            if (ready && published != ~size_t(0)) {
                bulk_wait_group<0>();
                __threadfence();
                fence_proxy_async_global();
                flag_release(ready + published, 1u);
                published = ~size_t(0);
            }
        }
        if (tid == 0 && ok) {
            tc_fence_after();
            mma_panels<true>(tmem, smem_u32(sm.qt), 16384, smem_u32(sm.dt), 16384, 8,
                             idesc_tf32_f32(128, 128), false);
            mma_commit(&sm.bar_mma);
            bulk_s2g(mt_img + item * (size_t)(2 * 16384), sm.mt, 2 * 16384);
            bulk_s2g(glv + item * AD, sm.gl[phase], AD * 4);
            bulk_commit_group();
        }
        if (ok) ok = mbar_wait_bounded(&sm.bar_mma, phase, kAWait);
        ok = __all_sync(0xffffffffu, ok);
        phase ^= 1u;
        tc_fence_after();
        if (ok) {
            // warp w: TMEM lanes 32 (w % 4).., columns 64 (w / 4)..: X rows, two tiles
            const int quad = warp & 3, half = warp >> 2, d = quad * 32 + (tid & 31);
            float v[32];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int vt = half * 2 + t;
                tmem_ld32(tmem_addr(tmem, quad * 32, vt * 32), v);
                float *dst = x_tiles + ((item * 4 + vt) * AD + d) * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) =
                        make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
        // the copies out have read the staging before the next item rewrites it
        if (tid == 0) {
            bulk_wait_group_read<0>();
            published = item;
        }
        tc_fence_before();
        // one verdict per CTA: after a wait that gave up, it stops
        if (__syncthreads_or(!ok)) break;
        k = k_next;
    }
    if (tid == 0) {
        if (!ok) {
            atomicExch(status, (int)KDA_ERR_TIMEOUT);
            // inputs requested for an item that will not run land first
            (void)mbar_wait_bounded(&sm.bar_in, phase, kAWait);
        }
        bulk_wait_group<0>();
        if (ok && ready && published != ~size_t(0)) {
            __threadfence();
            fence_proxy_async_global();
            flag_release(ready + published, 1u);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

constexpr int RD = 128, RC = 64, RBV = 32, RNT = RD / RBV, RSTAGE = 2;
constexpr uint32_t MT_BYTES = RD * RD * 2;   // -M'^T, bf16, 2 K-major panels
constexpr uint32_t SB_BYTES = RBV * RD * 2;   // dS_{c+1} operand, bf16, 2 K-major panels
constexpr uint32_t XT_BYTES = RD * RBV * 4;
constexpr uint32_t DS_IMG = RBV * RD * 4;
constexpr uint32_t GL_BYTES = RD * 4;
constexpr int kRThreads = 256;
constexpr uint32_t kRTmemCols = 2 * RBV;  // D2 ping-pong
constexpr long long kRWait = 2000000000LL;

struct RScanSmem {
    uint8_t mt[RSTAGE][MT_BYTES];  // 1024-aligned: offsets 0, 32 KB
    uint8_t sb[2][SB_BYTES];       // 64 KB, 72 KB
    float xs[RSTAGE][RD * RBV];
    float gl[RSTAGE][RD];
    uint64_t full[RSTAGE];   // stage loaded (bulk copies -> issuer, compute)
    uint64_t empty[RSTAGE];  // stage consumed: MMA commit + 128 compute threads
    uint64_t ready_s;        // dS operand written (compute -> issuer)
    uint64_t mma_s;          // product complete (commit -> compute)
    uint32_t tmem;
    volatile int32_t issued;
    volatile int32_t abort_flag;
};
constexpr size_t kRSmem = sizeof(RScanSmem) + 1024;
static_assert(kRSmem <= 227 * 1024, "reverse scan shared memory");
static_assert(offsetof(RScanSmem, sb) % 1024 == 0, "operand images 1024-aligned");

__device__ __forceinline__ bool rbarrier_or(bool pred) {
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

__global__ void __launch_bounds__(kRThreads, 1)
chunk_rscan_kernel(const uint8_t *__restrict__ mt_img, const float *__restrict__ x_tiles,
                   const float *__restrict__ glv, const float *__restrict__ d_final,
                   uint8_t *__restrict__ ds_img, uint8_t *__restrict__ ds_nat,
                   float *__restrict__ d_initial,
                   const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off,
                   int32_t N, int32_t T, int32_t H, const uint32_t *__restrict__ ready,
                   int *status) {
    extern __shared__ uint8_t smem_raw[];
    RScanSmem &sm = *reinterpret_cast<RScanSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t seq = blockIdx.x / RNT, vt = blockIdx.x % RNT, h = blockIdx.y;
    if (seq >= N) return;
    int32_t ta = 0, tb = T;
    if (cu) {
        ta = min(max(cu[seq], 0), T);
        tb = min(max(cu[seq + 1], ta), T);
    }
    const int32_t n_chunks = (tb - ta + RC - 1) / RC;
    const int32_t c_begin = chunk_off[seq];
    const size_t st_off = (((size_t)seq * H + h) * RD + (tid & 127)) * RD + (size_t)vt * RBV;

    float dS[RBV];
    if (tid < 128 && d_final) {
#pragma unroll
        for (int j = 0; j < RBV; j += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(d_final + st_off + j);
            dS[j] = x.x; dS[j + 1] = x.y; dS[j + 2] = x.z; dS[j + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < RBV; ++j) dS[j] = 0.f;
    }

    bool ok = true;
    if (n_chunks > 0) {
        if (tid == 0) {
            for (int i = 0; i < RSTAGE; ++i) {
                mbar_init(&sm.full[i], 1);
                mbar_init(&sm.empty[i], 1 + 128);
            }
            mbar_init(&sm.ready_s, 128);
            mbar_init(&sm.mma_s, 1);
            sm.issued = 0;
            sm.abort_flag = 0;
            fence_mbar_init();
        }
        if (warp == 0) {
            tmem_alloc(&sm.tmem, kRTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = sm.tmem;
        constexpr uint32_t IDESC = idesc_bf16_f32(128, RBV);  // A and B K-major
        // step n processes chunk c = c_begin + n_chunks - 1 - n
        auto item_of = [&](int32_t n) {
            return (size_t)(c_begin + n_chunks - 1 - n) * H + h;
        };

        if (warp == 4) {
            // -------- producer: -M'^T, the X tile and gl of each chunk --------
            if (lane == 0) {
                for (int32_t n = 0; n < n_chunks; ++n) {
                    const int stg = n % RSTAGE;
                    if (n >= RSTAGE) {
                        if (!mbar_wait_bounded(&sm.empty[stg], (uint32_t)(n / RSTAGE - 1) & 1u,
                                               kRWait) ||
                            sm.abort_flag) {
                            sm.abort_flag = 1;
                            break;
                        }
                    }
                    const size_t item = item_of(n);
                    // with flags: the item's inputs are published by the running
                    // producer kernel
                    if (ready) {
                        if (!flag_wait_bounded(ready + item, kRWait)) {
                            sm.abort_flag = 1;
                            break;
                        }
                        fence_proxy_async_global();
                    }
                    mbar_arrive_expect_tx(&sm.full[stg], MT_BYTES + XT_BYTES + GL_BYTES);
                    bulk_g2s(sm.mt[stg], mt_img + item * MT_BYTES, MT_BYTES, &sm.full[stg]);
                    bulk_g2s(sm.xs[stg], x_tiles + (item * RNT + vt) * (size_t)(RD * RBV),
                             XT_BYTES, &sm.full[stg]);
                    bulk_g2s(sm.gl[stg], glv + item * RD, GL_BYTES, &sm.full[stg]);
                    sm.issued = n + 1;
                }
            }
            __syncwarp();
        } else if (warp == 5) {
            // -------- MMA issuer: D2[n & 1] = (-M'^T) dS_{c+1} --------
            if (lane == 0) {
                int32_t done = 0;
                for (int32_t n = 0; n < n_chunks; ++n) {
                    const int stg = n % RSTAGE;
                    const bool got =
                        mbar_wait_bounded(&sm.full[stg], (uint32_t)(n / RSTAGE) & 1u, kRWait) &&
                        mbar_wait_bounded(&sm.ready_s, (uint32_t)n & 1u, kRWait);
                    if (!got || sm.abort_flag) {
                        sm.abort_flag = 1;
                        break;
                    }
                    tc_fence_after();
                    mma_panels<false>(tmem + (uint32_t)(n & 1) * RBV, smem_u32(sm.mt[stg]), 16384,
                                      smem_u32(sm.sb[n & 1]), 4096, 8, IDESC, false);
                    mma_commit(&sm.mma_s);
                    mma_commit(&sm.empty[stg]);
                    done = n + 1;
                }
                // every product issued is complete before TMEM and the shared
                // memory go away (they complete in order: wait for the last)
                if (done > 0 &&
                    !mbar_wait_bounded(&sm.mma_s, (uint32_t)(done - 1) & 1u, kRWait))
                    sm.abort_flag = 1;
            }
            __syncwarp();
        } else if (warp >= 6) {
            // (no role: the dS images leave from the compute threads' registers)
        } else {
            // -------- compute: thread = key row k --------
            const int k = tid;
            // dS_{c+1} of step n out as row k of panel vt of the K-major
            // (value-contiguous) image: the exact fp32 values, 128-byte
            // swizzled.  Issued while the step's product runs: before the
            // operand's proxy fence these stores would hold the fence up.
            auto put_global = [&](int32_t n) {
                if (!ds_nat) return;
                uint8_t *dst = ds_nat + item_of(n) * (size_t)(RD * RD * 4) + (size_t)vt * (RD * 128);
#pragma unroll
                for (int j = 0; j < RBV; j += 4)
                    *reinterpret_cast<float4 *>(dst + sw128_chunk(k, j >> 2)) =
                        make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
            };
            // ... and as rows 32 vt .. of the item's four 128-row panels of
            // dS^T (rows v, K = 32 keys each), tf32-rounded: the gradient
            // pass's operand image
            auto put_global_t = [&](int32_t n) {
                if (!ds_img) return;
                uint8_t *dst = ds_img + item_of(n) * (size_t)(RNT * DS_IMG) +
                               (size_t)(k >> 5) * (RNT * DS_IMG / 4);
#pragma unroll
                for (int j = 0; j < RBV; ++j)
                    *reinterpret_cast<float *>(dst + sw128_offset_f32(vt * RBV + j, k & 31)) =
                        tf32_operand(dS[j]);
            };
            // the product's B operand: dS_{c+1} as bf16 (fp32 range), rows v,
            // K = keys, two 64-key panels
            auto put_state = [&](int32_t n) {
                uint8_t *img = sm.sb[n & 1] + (k >> 6) * 4096u;
#pragma unroll
                for (int j = 0; j < RBV; ++j)
                    *reinterpret_cast<__nv_bfloat16 *>(img + sw128_offset(j, k & 63)) =
                        __float2bfloat16_rn(dS[j]);
                fence_proxy_async();
            };
            put_state(0);
            for (int32_t n = 0; n < n_chunks; ++n) {
                if (rbarrier_or(sm.abort_flag != 0)) break;
                tc_fence_before();
                mbar_arrive(&sm.ready_s);
                put_global(n);
                put_global_t(n);
                const int stg = n % RSTAGE;
                if (!mbar_wait_bounded(&sm.full[stg], (uint32_t)(n / RSTAGE) & 1u, kRWait))
                    sm.abort_flag = 1;
                const float g = sm.gl[stg][k];
                float x[RBV];
#pragma unroll
                for (int j = 0; j < RBV; j += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(&sm.xs[stg][k * RBV + j]);
                    x[j] = v.x; x[j + 1] = v.y; x[j + 2] = v.z; x[j + 3] = v.w;
                }
                mbar_arrive(&sm.empty[stg]);
                if (!mbar_wait_bounded(&sm.mma_s, (uint32_t)n & 1u, kRWait)) sm.abort_flag = 1;
                tc_fence_after();
                {
                    float d2[32];
                    tmem_ld32(tmem_addr(tmem + (uint32_t)(n & 1) * RBV, warp * 32, 0), d2);
#pragma unroll
                    for (int j = 0; j < RBV; ++j) dS[j] = fmaf(g, dS[j], d2[j] + x[j]);
                }
                // sb[(n + 1) & 1] held step n - 1's operand, whose product is done
                if (n + 1 < n_chunks) put_state(n + 1);
            }
        }
        __syncthreads();
        if (sm.abort_flag) {
            ok = false;
            if (tid == 0) {
                atomicExch(status, (int)KDA_ERR_TIMEOUT);
                const int32_t iss = sm.issued;
                for (int32_t j = max(iss - RSTAGE, 0); j < iss; ++j)
                    (void)mbar_wait_bounded(&sm.full[j % RSTAGE], (uint32_t)(j / RSTAGE) & 1u,
                                            kRWait);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, kRTmemCols);
        if (!ok) return;
    }
    if (d_initial && tid < 128) {
#pragma unroll
        for (int j = 0; j < RBV; j += 4)
            *reinterpret_cast<float4 *>(d_initial + st_off + j) =
                make_float4(dS[j], dS[j + 1], dS[j + 2], dS[j + 3]);
    }
    // launched beside its producer: this grid completes only after it, so
    // that later work in the stream sees everything both wrote
    if (tid == 0) pdl_wait_primaries();
}


size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct ChunkBwdLayout {
    size_t fwd, aux, mt, x, gl, ds_t, ds_n, img, ready, total;
};

ChunkBwdLayout chunk_bwd_layout(int32_t N, int32_t T, int32_t H) {
    const size_t maxc = (size_t)T / 64 + (size_t)N + 1, items = maxc * H;
    ChunkBwdLayout L;
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off += align256(n);
        return o;
    };
    L.fwd = take(chunk_tc_workspace_bytes(N, T, H));
    L.aux = take(items * kBwdAuxBytes);
    L.mt = take(items * MT_BYTES);
    L.x = take(items * RNT * (size_t)XT_BYTES);
    L.gl = take(items * AD * 4);
    L.ds_t = take(items * RNT * (size_t)DS_IMG);
    L.ds_n = take(items * AD * AD * 4);
    L.img = take(items * (size_t)kGradImgBytes);
    L.ready = take(items * sizeof(uint32_t));
    L.total = off;
    return L;
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int32_t N, int32_t T, int32_t H) {
    return chunk_bwd_layout(N, T, H).total;
}

cudaError_t launch_chunk_bwd(const BwdArgs &a, int *status, cudaStream_t stream) {
    if (a.D != AD || a.dtype != KDA_DTYPE_BF16 || !a.workspace) return cudaErrorInvalidValue;
    if (a.T == 0) {
        // no tokens: the initial-state gradient is the final-state gradient
        if (a.d_initial_state) {
            const size_t n = (size_t)a.N * a.H * AD * AD * sizeof(float);
            return a.d_final_state ? cudaMemcpyAsync(a.d_initial_state, a.d_final_state, n,
                                                     cudaMemcpyDeviceToDevice, stream)
                                   : cudaMemsetAsync(a.d_initial_state, 0, n, stream);
        }
        return cudaSuccess;
    }
    const ChunkBwdLayout L = chunk_bwd_layout(a.N, a.T, a.H);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    // 1. the forward engine, for its images (no outputs), keeping A^kk, A^qk
    StageClock clock;
    ChunkArgs f = {};
    f.q = a.q; f.k = a.k; f.v = a.v; f.log_alpha = a.log_alpha; f.beta = a.beta;
    f.scale = a.scale; f.initial_state = a.initial_state; f.cu_seqlens = a.cu_seqlens;
    f.out = nullptr; f.final_state = nullptr;
    f.N = a.N; f.T = a.T; f.H = a.H; f.D = AD; f.C = 64; f.G = 1; f.pro = 0;
    f.gbias = nullptr; f.galog = nullptr; f.dtype = KDA_DTYPE_BF16; f.out_f32 = 0;
    f.status = status; f.clock = &clock;
    f.bwd_aux = ws + L.aux;
    f.skip_out = 1;
    cudaError_t e = launch_chunk_tc(f, ws + L.fwd, L.aux - L.fwd, stream);
    if (e != cudaSuccess) return e;
    const ChunkScratchView view = chunk_tc_scratch_view(ws + L.fwd, a.N, a.T, a.H);
    const size_t maxc = view.max_chunks, items = maxc * a.H;
    // 2. -M'^T, X_c and exp(G_last) per (chunk, head)
    e = cudaFuncSetAttribute(chunk_bwd_aux_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kAuxSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_rscan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kRSmem);
    if (e != cudaSuccess) return e;
    AuxMaps amaps;
    memset(&amaps, 0, sizeof(amaps));
    if (a.d_out &&
        !encode_tile_map(&amaps.d, a.d_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H))
        return cudaErrorInvalidValue;
    // Beside each other when the reverse scan's CTAs fit in half of the SMs:
    // the persistent aux grid takes the others, publishes every item with a
    // flag, and the reverse scan (a programmatic dependent, so it starts only
    // once every aux CTA runs) follows the flags.  Otherwise one after the
    // other.
    const size_t rscan_ctas = (size_t)a.N * RNT * (size_t)a.H;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    const bool beside = sms > 0 && 2 * rscan_ctas <= (size_t)sms && !sequential_order_forced();
    const size_t aux_ctas = std::max<size_t>(
        1, std::min<size_t>(items, beside ? (size_t)sms - rscan_ctas
                                          : (size_t)std::max(sms, 1)));
    uint32_t *ready = beside ? reinterpret_cast<uint32_t *>(ws + L.ready) : nullptr;
    if (ready) {
        e = cudaMemsetAsync(ready, 0, items * sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    chunk_bwd_aux_kernel<<<(unsigned)aux_ctas, 256, kAuxSmem, stream>>>(
        amaps, view.img, view.chunk_tok, a.d_out != nullptr ? 1 : 0, ws + L.mt,
        reinterpret_cast<float *>(ws + L.x), reinterpret_cast<float *>(ws + L.gl), a.H,
        (int32_t)maxc, ready, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // 3. the reverse scan
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.N * RNT), (unsigned)a.H);
    cfg.blockDim = dim3((unsigned)kRThreads);
    cfg.dynamicSmemBytes = kRSmem;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = beside ? 1u : 0u;
    e = cudaLaunchKernelEx(&cfg, chunk_rscan_kernel, (const uint8_t *)(ws + L.mt),
                           reinterpret_cast<const float *>(ws + L.x),
                           reinterpret_cast<const float *>(ws + L.gl), a.d_final_state,
                           ws + L.ds_t, ws + L.ds_n, a.d_initial_state, a.cu_seqlens,
                           view.chunk_off, a.N, a.T, a.H, (const uint32_t *)ready, status);
    if (e != cudaSuccess) return e;
    // 4. every chunk's gradients from S_c and dS_{c+1}
    ChunkGradArgs g;
    g.chunk_tok = view.chunk_tok;
    g.n_items = items;
    g.T = a.T;
    g.H = a.H;
    g.scale = a.scale;
    g.aux = ws + L.aux;
    g.sst = view.sst;
    g.ds_t = ws + L.ds_t;
    g.ds_n = ws + L.ds_n;
    g.q = a.q; g.k = a.k; g.v = a.v; g.d_out = a.d_out;
    g.log_alpha = a.log_alpha; g.beta = a.beta;
    g.dq = a.dq; g.dk = a.dk; g.dv = a.dv; g.dlog_alpha = a.dlog_alpha; g.dbeta = a.dbeta;
    g.img = ws + L.img;
    g.status = status;
    return launch_chunk_grad(g, stream);
}

}  // namespace kda
