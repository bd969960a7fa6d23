// kda_api.cu -- the C ABI of libkda: host validation, engine selection,
// scratch handling and launch.  See include/kda.h for the contract.
#include <cmath>
#include <cstdint>

#include "kda_internal.cuh"

namespace kda {

namespace {

// Device-side status word, one per device that loaded the library.  Kernels
// with a bounded wait store KDA_ERR_TIMEOUT into it when the wait gives up;
// kda_device_status() reads and clears it.
__device__ int g_device_status = 0;

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices] = {};

// Device address of g_device_status on the current device (looked up once
// per device; the host-side symbol itself is not a device address).
int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool supported_dim(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128; }

int32_t default_chunk(int32_t d) { return d >= 64 ? 64 : 16; }

// Value heads (HV) and the group size HV / H.
int32_t value_heads(const kdaShape_t *s) { return s->num_v_heads ? s->num_v_heads : s->num_heads; }
int32_t group_size(const kdaShape_t *s) { return value_heads(s) / s->num_heads; }

// Shared shape checks.  Returns KDA_SUCCESS or the first error found.
kdaStatus_t check_shape(const kdaShape_t *s, bool step) {
    if (!s) return KDA_ERR_INVALID_ARG;
    if (s->num_seqs < 1 || s->total_tokens < 0 || s->num_heads < 1)
        return KDA_ERR_INVALID_ARG;
    if (s->num_v_heads < 0 || (s->num_v_heads % s->num_heads) != 0) return KDA_ERR_INVALID_ARG;
    if (s->prologue & ~(KDA_PROLOGUE_L2NORM_QK | KDA_PROLOGUE_BETA_LOGITS | KDA_PROLOGUE_GATE))
        return KDA_ERR_INVALID_ARG;
    if ((s->prologue & KDA_PROLOGUE_GATE) &&
        (!s->gate_bias || !s->gate_A_log || !aligned4(s->gate_bias) || !aligned4(s->gate_A_log)))
        return KDA_ERR_INVALID_ARG;
    if (s->d_k < 1 || s->d_v < 1) return KDA_ERR_INVALID_ARG;
    if (s->dtype != KDA_DTYPE_BF16 && s->dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (s->out_f32 != 0 && s->out_f32 != 1) return KDA_ERR_INVALID_ARG;
    if (step && s->total_tokens != s->num_seqs) return KDA_ERR_INVALID_ARG;
    if (!step) {
        if (s->chunk_size != 0 && s->chunk_size != 16 && s->chunk_size != 32 &&
            s->chunk_size != 64)
            return KDA_ERR_INVALID_ARG;
        if (s->engine < KDA_ENGINE_AUTO || s->engine > KDA_ENGINE_SIMT)
            return KDA_ERR_INVALID_ARG;
    }
    if (s->d_k != s->d_v || !supported_dim(s->d_k)) return KDA_ERR_UNSUPPORTED;
    if (value_heads(s) > 65535) return KDA_ERR_UNSUPPORTED;  // heads index grid.y
    // Index arithmetic inside the kernels is 64-bit, but token and
    // (token, head) counts travel as int32.
    if ((int64_t)s->total_tokens * value_heads(s) > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if ((int64_t)s->num_seqs * value_heads(s) > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    return KDA_SUCCESS;
}

bool tc_eligible(const kdaShape_t *s, int32_t C) {
    return s->dtype == KDA_DTYPE_BF16 && s->d_k == 128 && s->d_v == 128 && C == 64;
}

struct Plan {
    ChunkArgs args;
    bool use_tc;
    size_t workspace;
};

kdaStatus_t plan_chunk(const void *q, const void *k, const void *v, const float *log_alpha,
                       const float *beta, float scale, const float *initial_state,
                       const int32_t *cu_seqlens, void *out, float *final_state,
                       const kdaShape_t *shape, Plan *plan) {
    kdaStatus_t st = check_shape(shape, false);
    if (st != KDA_SUCCESS) return st;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && shape->num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > 0) {
        const void *vec[] = {q, k, v, out};
        for (const void *p : vec)
            if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
        const void *sc[] = {log_alpha, beta};
        for (const void *p : sc)
            if (!p || !aligned4(p)) return KDA_ERR_INVALID_ARG;
    }
    const void *opt[] = {initial_state, final_state};
    for (const void *p : opt)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned4(cu_seqlens)) return KDA_ERR_INVALID_ARG;
    const int32_t C = shape->chunk_size ? shape->chunk_size : default_chunk(shape->d_k);
    bool use_tc;
    switch (shape->engine) {
        case KDA_ENGINE_TENSOR:
            if (!tc_eligible(shape, C)) return KDA_ERR_UNSUPPORTED;
            use_tc = true;
            break;
        case KDA_ENGINE_SIMT: use_tc = false; break;
        default: use_tc = tc_eligible(shape, C); break;
    }
    // The tensor-core engine reads log_alpha through a TMA tensor map, whose
    // base must be 16-byte aligned.
    if (use_tc && shape->total_tokens > 0 && !aligned16(log_alpha)) return KDA_ERR_INVALID_ARG;
    ChunkArgs &a = plan->args;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens; a.out = out;
    a.final_state = final_state;
    a.N = shape->num_seqs; a.T = shape->total_tokens; a.H = value_heads(shape);
    a.G = group_size(shape); a.D = shape->d_k; a.C = C; a.dtype = shape->dtype;
    a.pro = shape->prologue; a.gbias = shape->gate_bias; a.galog = shape->gate_A_log;
    a.out_f32 = (shape->dtype == KDA_DTYPE_F32) ? 1 : shape->out_f32;
    plan->use_tc = use_tc;
    plan->workspace = use_tc ? chunk_tc_workspace_bytes(a.N, a.T, a.H) : 0;
    return KDA_SUCCESS;
}

kdaStatus_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KDA_SUCCESS;
    (void)cudaGetLastError();  // clear a non-sticky error so later calls start clean
    return KDA_ERR_CUDA;
}

kdaStatus_t run_plan(Plan p, void *workspace, cudaStream_t stream, StageClock *clock,
                     int32_t withhold_prep = 0, long long wait_cycles = 0) {
    StageClock local;
    p.args.diag_withhold_prep = withhold_prep;
    p.args.wait_cycles = wait_cycles;
    p.args.clock = clock ? clock : &local;
    p.args.status = device_status_ptr();
    if (!p.args.status) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    p.args.clock->mark(stream);
    if (p.use_tc) return cuda_status(launch_chunk_tc(p.args, workspace, p.workspace, stream));
    return cuda_status(launch_chunk_simt(p.args, stream));
}

// Device scratch of kda_chunk_fwd_host: the device copies of every input and
// output, then the engine's workspace, each region 256-byte aligned.
struct HostLayout {
    size_t q, k, v, la, beta, cu, s0, out, sf, gb, ga, ws, total;       // offsets
    size_t bq, bk, bv, bla, bbeta, bcu, bs, bout, bgb, bga;             // bytes
};

kdaStatus_t host_layout(const kdaShape_t *s, HostLayout *L) {
    kdaStatus_t st = check_shape(s, false);
    if (st != KDA_SUCCESS) return st;
    size_t ws = 0;
    st = kda_chunk_fwd_workspace_size(s, &ws);
    if (st != KDA_SUCCESS) return st;
    const size_t T = (size_t)s->total_tokens, H = (size_t)s->num_heads,
                 HV = (size_t)value_heads(s), dk = (size_t)s->d_k, dv = (size_t)s->d_v,
                 N = (size_t)s->num_seqs;
    const size_t es = s->dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t eo = (s->dtype == KDA_DTYPE_F32 || s->out_f32) ? 4 : 2;
    const bool gate = (s->prologue & KDA_PROLOGUE_GATE) != 0;
    L->bq = T * H * dk * es;
    L->bk = L->bq;
    L->bv = T * HV * dv * es;
    L->bla = T * HV * dk * 4;
    L->bbeta = T * HV * 4;
    L->bcu = (N + 1) * 4;
    L->bs = N * HV * dk * dv * 4;
    L->bout = T * HV * dv * eo;
    L->bgb = gate ? HV * dk * 4 : 0;
    L->bga = gate ? HV * 4 : 0;
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off += (n + 255) & ~size_t(255);
        return o;
    };
    L->q = take(L->bq);
    L->k = take(L->bk);
    L->v = take(L->bv);
    L->la = take(L->bla);
    L->beta = take(L->bbeta);
    L->cu = take(L->bcu);
    L->s0 = take(L->bs);
    L->out = take(L->bout);
    L->sf = take(L->bs);
    L->gb = take(L->bgb);
    L->ga = take(L->bga);
    L->ws = take(ws);
    L->total = off;
    return KDA_SUCCESS;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char *kda_status_string(kdaStatus_t status) {
    switch (status) {
        case KDA_SUCCESS: return "KDA_SUCCESS";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: outside the support matrix";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call or launch failed";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "KDA_ERR_UNKNOWN";
}

kdaStatus_t kda_chunk_fwd_workspace_size(const kdaShape_t *shape, size_t *bytes) {
    if (!bytes) return KDA_ERR_INVALID_ARG;
    kdaStatus_t st = check_shape(shape, false);
    if (st != KDA_SUCCESS) return st;
    const int32_t C = shape->chunk_size ? shape->chunk_size : default_chunk(shape->d_k);
    bool use_tc = shape->engine == KDA_ENGINE_SIMT ? false : tc_eligible(shape, C);
    if (shape->engine == KDA_ENGINE_TENSOR && !use_tc) return KDA_ERR_UNSUPPORTED;
    *bytes = use_tc ? chunk_tc_workspace_bytes(shape->num_seqs, shape->total_tokens,
                                               value_heads(shape))
                    : 0;
    return KDA_SUCCESS;
}

kdaStatus_t kda_chunk_fwd_ws_timed(const void *q, const void *k, const void *v,
                                   const float *log_alpha, const float *beta, float scale,
                                   const float *initial_state, const int32_t *cu_seqlens,
                                   void *out, float *final_state, const kdaShape_t *shape,
                                   void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream, cudaEvent_t *events,
                                   int32_t max_events, int32_t *n_recorded) {
    if (n_recorded) *n_recorded = 0;
    if (max_events < 0 || (max_events > 0 && !events)) return KDA_ERR_INVALID_ARG;
    Plan p;
    kdaStatus_t st = plan_chunk(q, k, v, log_alpha, beta, scale, initial_state, cu_seqlens,
                                out, final_state, shape, &p);
    if (st != KDA_SUCCESS) return st;
    if (p.workspace > 0) {
        if (!workspace || workspace_bytes < p.workspace) return KDA_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_INVALID_ARG;
    }
    StageClock clock;
    clock.events = events;
    clock.max_events = max_events;
    st = run_plan(p, workspace, stream, &clock);
    if (n_recorded) *n_recorded = clock.n < max_events ? clock.n : max_events;
    return st;
}

kdaStatus_t kda_chunk_fwd_ws(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta, float scale,
                             const float *initial_state, const int32_t *cu_seqlens,
                             void *out, float *final_state, const kdaShape_t *shape,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return kda_chunk_fwd_ws_timed(q, k, v, log_alpha, beta, scale, initial_state, cu_seqlens,
                                  out, final_state, shape, workspace, workspace_bytes, stream,
                                  nullptr, 0, nullptr);
}

kdaStatus_t kda_chunk_fwd_ws_diag(const void *q, const void *k, const void *v,
                                  const float *log_alpha, const float *beta, float scale,
                                  const float *initial_state, const int32_t *cu_seqlens,
                                  void *out, float *final_state, const kdaShape_t *shape,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t withhold_prep, int64_t wait_cycles,
                                  cudaStream_t stream) {
    Plan p;
    kdaStatus_t st = plan_chunk(q, k, v, log_alpha, beta, scale, initial_state, cu_seqlens,
                                out, final_state, shape, &p);
    if (st != KDA_SUCCESS) return st;
    if (!p.use_tc) return KDA_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < p.workspace ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KDA_ERR_INVALID_ARG;
    return run_plan(p, workspace, stream, nullptr, withhold_prep != 0 ? 1 : 0,
                    wait_cycles > 0 ? (long long)wait_cycles : 0);
}

kdaStatus_t kda_chunk_path_counts(uint64_t counts[3], cudaStream_t stream) {
    if (!counts) return KDA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return cuda_status(chunk_path_counts(counts, true));
}

kdaStatus_t kda_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, float scale, const float *initial_state,
                          const int32_t *cu_seqlens, void *out, float *final_state,
                          const kdaShape_t *shape, cudaStream_t stream) {
    Plan p;
    kdaStatus_t st = plan_chunk(q, k, v, log_alpha, beta, scale, initial_state, cu_seqlens,
                                out, final_state, shape, &p);
    if (st != KDA_SUCCESS) return st;
    void *ws = nullptr;
    if (p.workspace > 0) {
        if (cudaMallocAsync(&ws, p.workspace, stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return KDA_ERR_CUDA;
        }
    }
    st = run_plan(p, ws, stream, nullptr);
    if (ws && cudaFreeAsync(ws, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        if (st == KDA_SUCCESS) st = KDA_ERR_CUDA;
    }
    return st;
}

kdaStatus_t kda_chunk_fwd_host_scratch_size(const kdaShape_t *shape, size_t *bytes) {
    if (!bytes) return KDA_ERR_INVALID_ARG;
    HostLayout L;
    const kdaStatus_t st = host_layout(shape, &L);
    if (st != KDA_SUCCESS) return st;
    *bytes = L.total;
    return KDA_SUCCESS;
}

kdaStatus_t kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, float scale,
                               const float *initial_state, const int32_t *cu_seqlens,
                               void *out, float *final_state, const kdaShape_t *shape,
                               void *device_scratch, size_t scratch_bytes,
                               cudaStream_t stream) {
    HostLayout L;
    kdaStatus_t st = host_layout(shape, &L);
    if (st != KDA_SUCCESS) return st;
    if (!device_scratch || scratch_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(device_scratch) & 255u) != 0)
        return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && shape->num_seqs != 1) return KDA_ERR_INVALID_ARG;
    const bool any = shape->total_tokens > 0;
    if (any && (!q || !k || !v || !log_alpha || !beta || !out)) return KDA_ERR_INVALID_ARG;
    const bool gate = (shape->prologue & KDA_PROLOGUE_GATE) != 0;
    uint8_t *d = static_cast<uint8_t *>(device_scratch);
    cudaError_t e = cudaSuccess;
    auto h2d = [&](size_t off, const void *src, size_t n) {
        if (e == cudaSuccess && src && n > 0)
            e = cudaMemcpyAsync(d + off, src, n, cudaMemcpyHostToDevice, stream);
    };
    if (any) {
        h2d(L.q, q, L.bq);
        h2d(L.k, k, L.bk);
        h2d(L.v, v, L.bv);
        h2d(L.la, log_alpha, L.bla);
        h2d(L.beta, beta, L.bbeta);
    }
    h2d(L.cu, cu_seqlens, L.bcu);
    h2d(L.s0, initial_state, L.bs);
    if (gate) {
        h2d(L.gb, shape->gate_bias, L.bgb);
        h2d(L.ga, shape->gate_A_log, L.bga);
    }
    if (e != cudaSuccess) return cuda_status(e);
    kdaShape_t ds = *shape;  // the gate parameters, from their device copies
    if (gate) {
        ds.gate_bias = reinterpret_cast<const float *>(d + L.gb);
        ds.gate_A_log = reinterpret_cast<const float *>(d + L.ga);
    }
    Plan p;
    st = plan_chunk(d + L.q, d + L.k, d + L.v, reinterpret_cast<const float *>(d + L.la),
                    reinterpret_cast<const float *>(d + L.beta), scale,
                    initial_state ? reinterpret_cast<const float *>(d + L.s0) : nullptr,
                    cu_seqlens ? reinterpret_cast<const int32_t *>(d + L.cu) : nullptr,
                    d + L.out, final_state ? reinterpret_cast<float *>(d + L.sf) : nullptr, &ds,
                    &p);
    if (st != KDA_SUCCESS) return st;
    st = run_plan(p, d + L.ws, stream, nullptr);
    if (st != KDA_SUCCESS) return st;
    if (any) e = cudaMemcpyAsync(out, d + L.out, L.bout, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && final_state)
        e = cudaMemcpyAsync(final_state, d + L.sf, L.bs, cudaMemcpyDeviceToHost, stream);
    return cuda_status(e);
}

kdaStatus_t kda_recurrent_step(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta, float scale,
                               float *state, void *out, const kdaShape_t *shape,
                               cudaStream_t stream) {
    kdaStatus_t st = check_shape(shape, true);
    if (st != KDA_SUCCESS) return st;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    const void *vec[] = {q, k, v, state, out};
    for (const void *p : vec)
        if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const void *sc[] = {log_alpha, beta};
    for (const void *p : sc)
        if (!p || !aligned4(p)) return KDA_ERR_INVALID_ARG;
    StepArgs a;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.scale = scale;
    a.state = state; a.out = out; a.N = shape->num_seqs; a.H = value_heads(shape);
    a.G = group_size(shape);
    a.pro = shape->prologue; a.gbias = shape->gate_bias; a.galog = shape->gate_A_log;
    a.D = shape->d_k; a.dtype = shape->dtype;
    a.out_f32 = (shape->dtype == KDA_DTYPE_F32) ? 1 : shape->out_f32;
    return cuda_status(launch_recurrent_step(a, stream));
}

kdaStatus_t kda_recurrent_fwd(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta, float scale,
                              const int32_t *cu_seqlens, float *state_pool,
                              const int32_t *state_indices, int32_t num_slots, void *out,
                              const kdaShape_t *shape, cudaStream_t stream) {
    kdaStatus_t st = check_shape(shape, false);
    if (st != KDA_SUCCESS) return st;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && shape->num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (num_slots < 0 || (!state_indices && num_slots < shape->num_seqs))
        return KDA_ERR_INVALID_ARG;
    if ((int64_t)num_slots * value_heads(shape) > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (shape->total_tokens > 0) {
        const void *vec[] = {q, k, v, out, state_pool};
        for (const void *p : vec)
            if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
        const void *sc[] = {log_alpha, beta};
        for (const void *p : sc)
            if (!p || !aligned4(p)) return KDA_ERR_INVALID_ARG;
    }
    const void *idx[] = {cu_seqlens, state_indices};
    for (const void *p : idx)
        if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
    int *status = device_status_ptr();
    if (!status) return cuda_status(cudaErrorUnknown);
    RecurArgs a;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.scale = scale;
    a.cu_seqlens = cu_seqlens; a.state_indices = state_indices; a.num_slots = num_slots;
    a.pool = state_pool; a.out = out;
    a.N = shape->num_seqs; a.T = shape->total_tokens; a.H = value_heads(shape);
    a.G = group_size(shape); a.D = shape->d_k; a.dtype = shape->dtype;
    a.out_f32 = (shape->dtype == KDA_DTYPE_F32) ? 1 : shape->out_f32;
    a.pro = shape->prologue; a.gbias = shape->gate_bias; a.galog = shape->gate_A_log;
    a.status = status;
    return cuda_status(launch_recurrent_fwd(a, stream));
}

namespace {
kdaStatus_t check_conv(const kdaConvShape_t *s, bool step) {
    if (!s) return KDA_ERR_INVALID_ARG;
    if (s->num_seqs < 1 || s->channels < 1 || (!step && s->total_tokens < 0))
        return KDA_ERR_INVALID_ARG;
    if (s->dtype != KDA_DTYPE_BF16 && s->dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (s->activation != 0 && s->activation != 1) return KDA_ERR_INVALID_ARG;
    if (s->width < 2 || s->width > 8 || s->channels % 8 != 0) return KDA_ERR_UNSUPPORTED;
    if (s->num_seqs > 65535) return KDA_ERR_UNSUPPORTED;  // sequences index grid.y
    if ((int64_t)s->num_seqs * s->channels * s->width > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!step && (int64_t)s->total_tokens * s->channels > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    return KDA_SUCCESS;
}
}  // namespace

kdaStatus_t kda_short_conv_fwd(const void *x, const float *weight, const float *bias,
                               const int32_t *cu_seqlens, const void *cache_in, void *cache_out,
                               void *y, const kdaConvShape_t *shape, cudaStream_t stream) {
    kdaStatus_t st = check_conv(shape, false);
    if (st != KDA_SUCCESS) return st;
    if (!cu_seqlens && shape->num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (!weight || !aligned16(weight) || (bias && !aligned16(bias))) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > 0) {
        if (!x || !y || !aligned16(x) || !aligned16(y) || x == y) return KDA_ERR_INVALID_ARG;
    }
    const void *opt[] = {cache_in, cache_out, cu_seqlens};
    for (const void *p : opt)
        if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
    ConvArgs a;
    a.x = x; a.weight = weight; a.bias = bias; a.cu_seqlens = cu_seqlens;
    a.cache_in = cache_in; a.cache_out = cache_out; a.y = y;
    a.N = shape->num_seqs; a.T = shape->total_tokens; a.C = shape->channels;
    a.W = shape->width; a.dtype = shape->dtype; a.activation = shape->activation;
    a.step = false;
    return cuda_status(launch_short_conv(a, stream));
}

kdaStatus_t kda_short_conv_step(const void *x, const float *weight, const float *bias,
                                void *cache, void *y, const kdaConvShape_t *shape,
                                cudaStream_t stream) {
    kdaStatus_t st = check_conv(shape, true);
    if (st != KDA_SUCCESS) return st;
    const void *need[] = {x, weight, cache, y};
    for (const void *p : need)
        if (!p || !aligned4(p)) return KDA_ERR_INVALID_ARG;
    if (bias && !aligned4(bias)) return KDA_ERR_INVALID_ARG;
    ConvArgs a;
    a.x = x; a.weight = weight; a.bias = bias; a.cu_seqlens = nullptr;
    a.cache_in = cache; a.cache_out = cache; a.y = y;
    a.N = shape->num_seqs; a.T = shape->num_seqs; a.C = shape->channels;
    a.W = shape->width; a.dtype = shape->dtype; a.activation = shape->activation;
    a.step = true;
    return cuda_status(launch_short_conv(a, stream));
}

kdaStatus_t kda_recurrent_bwd(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta, float scale,
                              const float *initial_state, const int32_t *cu_seqlens,
                              const void *d_out, const float *d_final_state, float *dq, float *dk,
                              float *dv, float *dlog_alpha, float *dbeta, float *d_initial_state,
                              const kdaShape_t *shape, cudaStream_t stream) {
    kdaStatus_t st = check_shape(shape, false);
    if (st != KDA_SUCCESS) return st;
    if (group_size(shape) != 1 || shape->prologue != 0) return KDA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && shape->num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > 0) {
        const void *need[] = {q, k, v, log_alpha, beta, dq, dk, dv, dlog_alpha, dbeta};
        for (const void *p : need)
            if (!p || !aligned4(p)) return KDA_ERR_INVALID_ARG;
        if (d_out && !aligned4(d_out)) return KDA_ERR_INVALID_ARG;
    }
    const void *states[] = {initial_state, d_final_state, d_initial_state};
    for (const void *p : states)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned4(cu_seqlens)) return KDA_ERR_INVALID_ARG;
    BwdArgs a;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens; a.d_out = d_out;
    a.d_final_state = d_final_state; a.dq = dq; a.dk = dk; a.dv = dv; a.dlog_alpha = dlog_alpha;
    a.dbeta = dbeta; a.d_initial_state = d_initial_state;
    a.N = shape->num_seqs; a.T = shape->total_tokens; a.H = shape->num_heads;
    a.D = shape->d_k; a.dtype = shape->dtype;
    const size_t bytes = recurrent_bwd_workspace_bytes(a.N, a.T, a.H, a.D);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    a.workspace = ws;
    const cudaError_t e = launch_recurrent_bwd(a, stream);
    const cudaError_t f = cudaFreeAsync(ws, stream);
    return cuda_status(e != cudaSuccess ? e : f);
}

namespace {
// Arguments of kda_chunk_bwd / kda_chunk_bwd_ws, checked before anything runs.
kdaStatus_t plan_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                           const float *beta, float scale, const float *initial_state,
                           const int32_t *cu_seqlens, const void *d_out,
                           const float *d_final_state, float *dq, float *dk, float *dv,
                           float *dlog_alpha, float *dbeta, float *d_initial_state,
                           const kdaShape_t *shape, BwdArgs &a) {
    kdaStatus_t st = check_shape(shape, false);
    if (st != KDA_SUCCESS) return st;
    if (group_size(shape) != 1 || shape->prologue != 0 || shape->dtype != KDA_DTYPE_BF16 ||
        shape->d_k != 128)
        return KDA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && shape->num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (shape->total_tokens > 0) {
        // the forward engine's tensor maps want 16-byte aligned q, k, v, log_alpha
        const void *need16[] = {q, k, v, log_alpha};
        for (const void *p : need16)
            if (!p || !aligned16(p)) return KDA_ERR_INVALID_ARG;
        const void *need[] = {beta, dq, dk, dv, dlog_alpha, dbeta};
        for (const void *p : need)
            if (!p || !aligned4(p)) return KDA_ERR_INVALID_ARG;
        if (d_out && !aligned4(d_out)) return KDA_ERR_INVALID_ARG;
    }
    const void *states[] = {initial_state, d_final_state, d_initial_state};
    for (const void *p : states)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned4(cu_seqlens)) return KDA_ERR_INVALID_ARG;
    a.q = q; a.k = k; a.v = v; a.log_alpha = log_alpha; a.beta = beta; a.scale = scale;
    a.initial_state = initial_state; a.cu_seqlens = cu_seqlens; a.d_out = d_out;
    a.d_final_state = d_final_state; a.dq = dq; a.dk = dk; a.dv = dv; a.dlog_alpha = dlog_alpha;
    a.dbeta = dbeta; a.d_initial_state = d_initial_state;
    a.N = shape->num_seqs; a.T = shape->total_tokens; a.H = shape->num_heads;
    a.D = shape->d_k; a.dtype = shape->dtype;
    return KDA_SUCCESS;
}
}  // namespace

kdaStatus_t kda_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, float scale, const float *initial_state,
                          const int32_t *cu_seqlens, const void *d_out,
                          const float *d_final_state, float *dq, float *dk, float *dv,
                          float *dlog_alpha, float *dbeta, float *d_initial_state,
                          const kdaShape_t *shape, cudaStream_t stream) {
    BwdArgs a;
    const kdaStatus_t st = plan_chunk_bwd(q, k, v, log_alpha, beta, scale, initial_state,
                                          cu_seqlens, d_out, d_final_state, dq, dk, dv,
                                          dlog_alpha, dbeta, d_initial_state, shape, a);
    if (st != KDA_SUCCESS) return st;
    int *status = device_status_ptr();
    if (!status) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    const size_t bytes = chunk_bwd_workspace_bytes(a.N, a.T, a.H);
    void *ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    a.workspace = ws;
    const cudaError_t e = launch_chunk_bwd(a, status, stream);
    const cudaError_t f = cudaFreeAsync(ws, stream);
    return cuda_status(e != cudaSuccess ? e : f);
}

kdaStatus_t kda_chunk_bwd_workspace_size(const kdaShape_t *shape, size_t *bytes) {
    if (!bytes) return KDA_ERR_INVALID_ARG;
    kdaStatus_t st = check_shape(shape, false);
    if (st != KDA_SUCCESS) return st;
    if (group_size(shape) != 1 || shape->prologue != 0 || shape->dtype != KDA_DTYPE_BF16 ||
        shape->d_k != 128)
        return KDA_ERR_UNSUPPORTED;
    *bytes = chunk_bwd_workspace_bytes(shape->num_seqs, shape->total_tokens, shape->num_heads);
    return KDA_SUCCESS;
}

kdaStatus_t kda_chunk_bwd_ws(const void *q, const void *k, const void *v, const float *log_alpha,
                             const float *beta, float scale, const float *initial_state,
                             const int32_t *cu_seqlens, const void *d_out,
                             const float *d_final_state, float *dq, float *dk, float *dv,
                             float *dlog_alpha, float *dbeta, float *d_initial_state,
                             const kdaShape_t *shape, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    BwdArgs a;
    const kdaStatus_t st = plan_chunk_bwd(q, k, v, log_alpha, beta, scale, initial_state,
                                          cu_seqlens, d_out, d_final_state, dq, dk, dv,
                                          dlog_alpha, dbeta, d_initial_state, shape, a);
    if (st != KDA_SUCCESS) return st;
    if (!workspace || workspace_bytes < chunk_bwd_workspace_bytes(a.N, a.T, a.H) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return KDA_ERR_INVALID_ARG;
    int *status = device_status_ptr();
    if (!status) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    a.workspace = workspace;
    return cuda_status(launch_chunk_bwd(a, status, stream));
}

kdaStatus_t kda_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    int value = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbol(&value, g_device_status, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return value == 0 ? KDA_SUCCESS : static_cast<kdaStatus_t>(value);
}

}  // extern "C"
