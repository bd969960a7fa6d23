// tc_ptx.cuh -- hand-written inline PTX for the sm_103a tensor-core engine:
// mbarriers, bulk async copies (TMA engine, non-tensor form), TMEM
// allocation, tcgen05.mma (kind::f16, one CTA) and TMEM loads.
//
// Operand layout used everywhere: K-major, 128-byte swizzle.  A tile of R
// rows (R a multiple of 8) and 128 bytes of K (64 half-precision or 32 tf32
// elements) is a "panel": row r lives at byte r*128 of the panel, and its
// 16-byte chunk c sits at chunk position (c ^ (r % 8)).  Panels are
// 1024-byte aligned, so the swizzle the tensor core applies (address bits
// [4,7) xor bits [7,10)) matches.  The MMA walks K in 32-byte steps by
// advancing the descriptor start address inside the panel.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of element (row, col) in a K-major SW128 panel of bf16.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + ((col & 7u) << 1);
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row`.
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t row, uint32_t chunk) {
    return row * 128u + (((chunk ^ row) & 7u) << 4);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// `max_cycles` SM clocks.  Returns false when the limit is reached.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long max_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > max_cycles) return false;
    }
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched as a programmatic dependent
// may start before the kernel ahead of it in the stream has finished; it
// waits with pdl_wait_primaries() before touching that kernel's results
// (both are no-ops for an ordinary launch).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primaries() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// hand-off between CTAs of concurrently running kernels: the producer writes
// with bulk copies, waits for them, and publishes a flag with release
// semantics; the consumer acquires the flag before it reads with bulk copies.
// The proxy fences order the bulk-copy (async proxy) accesses against the
// flag's ordinary (generic proxy) access on each side.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void flag_release(uint32_t *f, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t flag_acquire(const uint32_t *f) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
// Spins (with a short sleep) until *f is non-zero or max_cycles have passed.
__device__ __forceinline__ bool flag_wait_bounded(const uint32_t *f, long long max_cycles) {
    if (flag_acquire(f)) return true;
    const long long t0 = clock64();
    while (true) {
        __nanosleep(100);
        if (flag_acquire(f)) return true;
        if (clock64() - t0 > max_cycles) return false;
    }
}

// ---------------------------------------------------------------------------
// bulk async copy global -> shared, completion counted on an mbarrier
// (addresses 16-byte aligned, size a multiple of 16)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// bulk async copy shared -> global, bulk-group completion (addresses 16-byte
// aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

// Tiled tensor load (TMA), 3-D coordinates {x innermost, y, z}; the tensor
// map lives in kernel parameter space (__grid_constant__).
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int32_t x, int32_t y,
                                            int32_t z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// Brings a 3-D tile into L2 only (a hint: no completion, no shared memory).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void *tmap, int32_t x, int32_t y,
                                                   int32_t z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Bulk prefetch of a contiguous global range into L2 (no completion to wait
// for: a hint).  Address and size multiples of 16 bytes.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Tiled tensor store (TMA) from shared memory, bulk-group completion.
__device__ __forceinline__ void tma_store_3d(const void *tmap, const void *src, int32_t x,
                                             int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(tmap)),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until every committed bulk group has completed (writes visible).
// Waits until at most N of this thread's most recent bulk groups are still
// writing (the older ones are complete).
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor core operand reads, bulk copies).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMEM
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address, 16 B units
    d |= static_cast<uint64_t>(1u) << 16;                   // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;           // stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                   // version
    d |= static_cast<uint64_t>(2u) << 61;                   // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp32 D, A and B K-major of one element format
// (0 = f16 or 1 = bf16 under kind::f16, 2 = tf32 under kind::tf32).
enum : uint32_t { kFmtF16 = 0, kFmtBF16 = 1, kFmtTF32 = 2 };
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t fmt, int M, int N) {
    return (1u << 4)                                   // D: f32
           | (fmt << 7)                                // A format
           | (fmt << 10)                               // B format
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return idesc_f32acc(kFmtBF16, M, N);
}
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return idesc_f32acc(kFmtF16, M, N);
}
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
    return idesc_f32acc(kFmtTF32, M, N);
}

// ---------------------------------------------------------------------------
// MMA and commit (issued by one thread)
// ---------------------------------------------------------------------------
// Half-precision operands (f16 or bf16, chosen by the instruction descriptor).
__device__ __forceinline__ void mma_half(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// tf32 operands (fp32 storage, 8 elements = 32 bytes per K step).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// D[128 x N] (+)= A[128 x K] * B[N x K]^T over SW128 panels, K walked in
// 32-byte steps (16 half-precision or 8 tf32 elements), 4 steps per panel.
// a_base/b_base: shared addresses of the first panel; panel strides in bytes.
template <bool TF32 = false>
__device__ __forceinline__ void mma_panels(uint32_t d_tmem, uint32_t a_base, uint32_t a_panel,
                                           uint32_t b_base, uint32_t b_panel, int ksteps,
                                           uint32_t idesc, bool accumulate_first) {
#pragma unroll
    for (int ks = 0; ks < ksteps; ++ks) {
        const uint32_t a = a_base + (ks >> 2) * a_panel + (ks & 3) * 32;
        const uint32_t b = b_base + (ks >> 2) * b_panel + (ks & 3) * 32;
        const uint32_t acc = (ks > 0 || accumulate_first) ? 1u : 0u;
        if (TF32)
            mma_tf32(d_tmem, sdesc_sw128(a), sdesc_sw128(b), idesc, acc);
        else
            mma_half(d_tmem, sdesc_sw128(a), sdesc_sw128(b), idesc, acc);
    }
}

// Half-precision A K-major (panels of 128-byte rows), B MN-major (N = 64,
// SW128: one 128-byte row of 64 values per K index): K walks 32 bytes of A
// and 16 rows = 2048 bytes of B per step.
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

// ---------------------------------------------------------------------------
// TMEM -> registers: 32 lanes x 32-bit, N consecutive columns per thread
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 32-column loads in flight together, one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&va)[32],
                                            float (&vb)[32]) {
    uint32_t r[32], q[32];
#define KDA_LD32(R, ADDR)                                                                   \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "                                  \
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"                  \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" \
                 : "=r"(R[0]), "=r"(R[1]), "=r"(R[2]), "=r"(R[3]), "=r"(R[4]), "=r"(R[5]),  \
                   "=r"(R[6]), "=r"(R[7]), "=r"(R[8]), "=r"(R[9]), "=r"(R[10]), "=r"(R[11]), \
                   "=r"(R[12]), "=r"(R[13]), "=r"(R[14]), "=r"(R[15]), "=r"(R[16]),         \
                   "=r"(R[17]), "=r"(R[18]), "=r"(R[19]), "=r"(R[20]), "=r"(R[21]),         \
                   "=r"(R[22]), "=r"(R[23]), "=r"(R[24]), "=r"(R[25]), "=r"(R[26]),         \
                   "=r"(R[27]), "=r"(R[28]), "=r"(R[29]), "=r"(R[30]), "=r"(R[31])          \
                 : "r"(ADDR))
    KDA_LD32(r, ta);
    KDA_LD32(q, tb);
#undef KDA_LD32
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(q[i]);
    }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Five loads of 8 consecutive columns each (any addresses), one wait.
__device__ __forceinline__ void tmem_ld8x5(const uint32_t (&ta)[5], float (&v)[5][8]) {
    uint32_t r[5][8];
#pragma unroll
    for (int k = 0; k < 5; ++k)
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[k][0]), "=r"(r[k][1]), "=r"(r[k][2]), "=r"(r[k][3]),
                       "=r"(r[k][4]), "=r"(r[k][5]), "=r"(r[k][6]), "=r"(r[k][7])
                     : "r"(ta[k]));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int k = 0; k < 5; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[k][i] = __uint_as_float(r[k][i]);
}

// registers -> TMEM: 32 lanes x 32-bit, 32 consecutive columns per thread
// (each warp writes its own 32-lane quadrant), then wait for the store.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
        "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
        "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// registers -> TMEM: one 32-bit column per thread (its lane), no wait (the
// caller issues tcgen05.wait::st before anything depends on the store).
__device__ __forceinline__ void tmem_st1_nowait(uint32_t taddr, float v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "f"(v)
                 : "memory");
}
// registers -> TMEM: 8 consecutive 32-bit columns per thread, no wait (the
// caller issues tcgen05.wait::st before anything depends on the stores).
__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// TMEM address of (lane, column): lane in bits [16, 32), column in [0, 16).
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// An fp32 value as a tf32 MMA operand (10-bit significand), rounded to nearest
// with ties away from zero.  A tcgen05 MMA of kind::tf32 reads only the top 19
// bits of each 32-bit operand and drops the other 13, so adding half a unit of
// the dropped bits (0x1000) to the bit pattern is the whole rounding: the sum
// carries into the kept bits exactly when the dropped part is at least half,
// and the tensor core's truncation does the rest (the outputs are bit-identical
// to those from operands with the low bits cleared as well).  The result is an
// MMA operand only, not an fp32 value: its low bits are left as they were.
// Finite inputs only (the operands here are finite).
__device__ __forceinline__ float tf32_operand(float x) {
    return __uint_as_float(__float_as_uint(x) + 0x1000u);
}

// 2^x with the SM's special-function unit (ex2.approx.ftz.f32 of the PTX ISA:
// relative error about 2^-22, results below 2^-126 flushed to zero).  The
// chunk engine keeps its cumulative log decays in base 2, so that every
// exp(a - b) it needs is ex2 of a difference.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): ln-domain -> base 2

// Byte offset of fp32 element (row, col) in a K-major SW128 panel (32 per row).
__device__ __forceinline__ uint32_t sw128_offset_f32(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 2) ^ row) & 7u) << 4) + ((col & 3u) << 2);
}

}  // namespace tc
}  // namespace kda
