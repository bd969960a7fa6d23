// kda_internal.cuh -- declarations shared by the libkda translation units.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kda.h"

namespace kda {

// Optional device-side stage timing: records caller-created events on the
// launch stream before the first kernel and after each kernel.
struct StageClock {
    cudaEvent_t *events = nullptr;
    int32_t max_events = 0;
    int32_t n = 0;
    void mark(cudaStream_t s) {
        if (events && n < max_events) cudaEventRecord(events[n], s);
        ++n;
    }
};

// Everything a chunk launch needs, after host validation.
struct ChunkArgs {
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    float scale;
    const float *initial_state;
    const int32_t *cu_seqlens;   // device, N + 1 entries, or nullptr (one sequence)
    void *out;
    float *final_state;
    int32_t N, T, H, D, C;      // H: value heads (v, log_alpha, beta, out, states)
    int32_t G;                   // value heads per q/k head (q, k have H / G heads)
    int32_t pro;                 // kdaPrologue_t bits
    const float *gbias, *galog;  // gate bias [H, D], sensitivity [H] (KDA_PROLOGUE_GATE)
    int32_t dtype;               // kdaDtype_t of q, k, v
    int32_t out_f32;             // 1: out is float32, 0: out has dtype
    int *status;                 // device status word (kernels with bounded waits
                                 // store KDA_ERR_TIMEOUT here when one gives up)
    StageClock *clock;           // never null inside the launchers
    int32_t diag_withhold_prep = 0;  // diagnostic: launch no prep (the scan's waits run out)
    long long wait_cycles = 0;       // limit of every bounded wait in SM clocks (0: default)
    // For the chunkwise backward (tensor-core engine only): when set, the prep
    // also stores every item's A^kk and A^qk (f16 K-major SW128 panels, 8 KB
    // each, kBwdAuxBytes per item at item * kBwdAuxBytes), and skip_out
    // leaves the output pass out (out may then be null).
    uint8_t *bwd_aux = nullptr;
    int32_t skip_out = 0;
};
constexpr uint32_t kBwdAuxBytes = 16384;

struct StepArgs {
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    float scale;
    float *state;
    void *out;
    int32_t N, H, D;            // H: value heads
    int32_t G;                  // value heads per q/k head
    int32_t pro;                // kdaPrologue_t bits
    const float *gbias, *galog;
    int32_t dtype;
    int32_t out_f32;
};

// Multi-token fused recurrent pass over packed sequences with a slot-indexed
// state pool (kda_decode.cu).
struct RecurArgs {
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    float scale;
    const int32_t *cu_seqlens;     // device [N + 1] or nullptr (one sequence)
    const int32_t *state_indices;  // device [N] or nullptr (slot = sequence)
    int32_t num_slots;
    float *pool;                   // [num_slots, H, D, D]
    void *out;
    int32_t N, T, H, D;            // H: value heads
    int32_t G;                     // value heads per q/k head
    int32_t pro;                   // kdaPrologue_t bits
    const float *gbias, *galog;
    int32_t dtype;
    int32_t out_f32;
    int *status;                   // device status word
};

// Gradients of the recurrence (kda_backward.cu).
struct BwdArgs {
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    float scale;
    const float *initial_state;    // [N, H, D, D] or nullptr
    const int32_t *cu_seqlens;
    const void *d_out;             // [T, H, D] dtype of q, or nullptr (zero)
    const float *d_final_state;    // [N, H, D, D] or nullptr (zero)
    float *dq, *dk, *dv, *dlog_alpha, *dbeta, *d_initial_state;
    void *workspace;               // recurrent_bwd_workspace_bytes, 256-byte aligned
    int32_t N, T, H, D, dtype;
};
size_t recurrent_bwd_workspace_bytes(int32_t N, int32_t T, int32_t H, int32_t D);
cudaError_t launch_recurrent_bwd(const BwdArgs &a, cudaStream_t stream);

// Chunkwise backward (kda_backward_chunk.cu): the forward engine's images, a
// reverse scan over chunks for the state gradient at every chunk boundary,
// then the recurrent walk per 64-token chunk from its boundary values.
// bf16, D = 128, no prologue, no value-head groups.
size_t chunk_bwd_workspace_bytes(int32_t N, int32_t T, int32_t H);
cudaError_t launch_chunk_bwd(const BwdArgs &a, int *status, cudaStream_t stream);

// The per-chunk gradient pass of the chunkwise backward
// (kda_backward_grad.cu), from what the forward engine, its A^kk / A^qk
// store and the reverse scan leave: two launches over the (chunk, head)
// items, bf16 q/k/v/dO, D = 128, C = 64.
struct ChunkGradArgs {
    const int2 *chunk_tok;        // [max chunks] first token, length
    size_t n_items;               // max chunks x H
    int32_t T, H;
    float scale;
    const uint8_t *aux;           // per item kBwdAuxBytes: A^kk, A^qk (f16 panels)
    const uint8_t *sst;           // per item 2 x 16 KB: S_c (f16, value tiles of 64)
    const uint8_t *ds_t;          // per item 4 x 16 KB: dS_{c+1}^T tf32 tiles of 32 rows
    const uint8_t *ds_n;          // per item 64 KB: dS_{c+1} fp32, K-major SW128 panels
    const void *q, *k, *v, *d_out;  // bf16 [T, H, 128] (d_out may be null)
    const float *log_alpha, *beta;
    float *dq, *dk, *dv, *dlog_alpha, *dbeta;
    uint8_t *img;                 // scratch, kGradImgBytes per item (the first kernel's
                                  // gradients as the second's operand images)
    int *status;
};
constexpr uint32_t kGradImgBytes = 96 * 1024;
cudaError_t launch_chunk_grad(const ChunkGradArgs &a, cudaStream_t stream);

// The fused input prologue, as each kernel applies it to one element.
constexpr float kL2Eps = 1e-6f;
// Packed fp32 pairs (sm_100 and later): one instruction for two IEEE fp32
// multiplies or fused multiply-adds, bit-identical to the scalar forms.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float pro_sigmoid(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
// gate logit g of channel j of a head with sensitivity exp(A_log) = sens and
// bias b[j] -> log retention -5 sigmoid(sens (g + b[j]))
__device__ __forceinline__ float pro_gate(float g, float sens, float bias) {
    return -5.f * pro_sigmoid(sens * (g + bias));
}

// Short causal convolution (kda_conv.cu).
struct ConvArgs {
    const void *x;                 // [T, C] (prefill) or [N, C] (step)
    const float *weight, *bias;    // [C, W], [C] or nullptr
    const int32_t *cu_seqlens;     // prefill: [N + 1] or nullptr (one sequence)
    const void *cache_in;          // prefill: [N, C, W] or nullptr (zeros)
    void *cache_out;               // prefill: [N, C, W] or nullptr; step: the cache, in place
    void *y;
    int32_t N, T, C, W, dtype, activation;
    bool step;
};
cudaError_t launch_short_conv(const ConvArgs &a, cudaStream_t stream);

// fp32 CUDA-core chunk engine (kda_chunk_simt.cu).  Needs no scratch.
cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t stream);

// Decode step and the multi-token recurrent pass (kda_decode.cu).
cudaError_t launch_recurrent_step(const StepArgs &a, cudaStream_t stream);
cudaError_t launch_recurrent_fwd(const RecurArgs &a, cudaStream_t stream);

// A [T, H, 128] row-major tensor as a 3-D tensor map {128, H, T} whose box
// is one head's [64 tokens x box_x channels] tile (rows past T read as zero),
// for tiled TMA loads (kda_chunk_tc.cu).
bool encode_tile_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t esize,
                     int32_t T, int32_t H, uint32_t box_x = 128,
                     CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE);
// KDA_LAUNCH_ORDER=sequential in the environment: every multi-kernel path
// runs its kernels one after another (kda_chunk_tc.cu).
bool sequential_order_forced();

// Tensor-core chunk engine (kda_chunk_tc.cu): bf16, D = 128, C = 64.
size_t chunk_tc_workspace_bytes(int32_t N, int32_t T, int32_t H);
// Items per path of the decayed products since the last clear (mid, half,
// direct), on the current device.
cudaError_t chunk_path_counts(uint64_t counts[3], bool clear);
cudaError_t launch_chunk_tc(const ChunkArgs &a, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);
// What a finished launch_chunk_tc leaves in its workspace, for the backward:
// per (chunk c, head h), item = c * H + h, chunks numbered sequence by
// sequence (chunk_off[s] = first chunk of sequence s; chunk_tok[c] = {first
// token, length}, length 0 past the last chunk; max_chunks entries):
//   img  + item * kChunkImgStride: f16 -M' (2 K-major panels of 128 rows at
//        0), Q' keys 0..63 / 64..127 (64 rows at 49152 / 65536), exp(G_last)
//        [128] f32 at 73728
//   sst  + (item * 2 + vt) * 16384: S_c entering the chunk, value columns
//        64 vt .. 64 vt + 63, f16, one 128-byte-swizzled row of 64 values
//        per key row
struct ChunkScratchView {
    const uint8_t *img;
    const uint8_t *sst;
    const int2 *chunk_tok;
    const int32_t *chunk_off;
    size_t max_chunks;
};
constexpr uint32_t kChunkImgStride = 74752;
ChunkScratchView chunk_tc_scratch_view(void *workspace, int32_t N, int32_t T, int32_t H);

}  // namespace kda
