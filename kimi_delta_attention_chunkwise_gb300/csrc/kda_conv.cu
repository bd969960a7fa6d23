// kda_conv.cu -- the short causal convolution of the KDA layer and its cache.
//
// "Linear Attention, From Scratch to Kimi 3", sec. 7: every channel owns a
// W-tap temporal filter (no mixing across channels; q, k and v each have
// their own), decode keeps a cache of each sequence's most recent
// pre-convolution inputs, and packed sequences (sec. 9) never see each
// other's tokens.  Output at token t of a sequence:
//     y[t, c] = act( sum_i w[c, i] * x[t - W + 1 + i, c] + bias[c] )
// with inputs before the sequence's first token taken from its cache (slot
// W - 1 the most recent) or zero.
//
// Memory-bound elementwise work: a thread owns one 16-byte vector of
// consecutive channels (8 bf16 or 4 fp32) for a block of TB tokens; it issues
// all of the block's rows and the W - 1 before them as independent loads
// first, then filters from registers, so every input row is read once per
// block (plus the halo) and every output written once, fully coalesced along
// channels.  Each row is unpacked once, into a window of the W most recent
// rows; a block with no sequence start inside its window (nearly all of them)
// takes a path with no per-tap boundary test.
#include <cstdint>
#include <cuda_bf16.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kConvThreads = 128;
constexpr int kConvTB = 8;   // tokens per thread
constexpr int kConvMinBlocks = 4;  // resident CTAs per SM (fewer registers spill)

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
    using Raw = float4;
    __device__ static Raw load_raw(const float *p) { return *reinterpret_cast<const float4 *>(p); }
    __device__ static Raw zero_raw() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ static void unpack(const Raw &x, float (&v)[4]) {
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
    __device__ static void store(float *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
// bf16: 8 channels (16 bytes) per thread
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    using Raw = uint4;
    __device__ static Raw load_raw(const __nv_bfloat16 *p) {
        return *reinterpret_cast<const uint4 *>(p);
    }
    __device__ static Raw zero_raw() { return make_uint4(0, 0, 0, 0); }
    __device__ static void unpack(const Raw &x, float (&v)[8]) {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&v)[8]) {
        uint4 x;
        uint32_t *w = &x.x;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(p) = x;
    }
};

// SiLU(z) = z * sigmoid(z); __fdividef returns 0 once the divisor passes
// 2^126, which is SiLU's limit for very negative z.
__device__ __forceinline__ float act(float z, int activation) {
    return activation ? __fdividef(z, 1.f + __expf(-z)) : z;
}

__device__ __forceinline__ int32_t seq_of(const int32_t *cu, int32_t N, int32_t t) {
    // largest s with cu[s] <= t (cu non-decreasing); cu == nullptr: one sequence
    if (!cu) return 0;
    int32_t lo = 0, hi = N - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads, kConvMinBlocks)
short_conv_fwd_kernel(const T *__restrict__ x, const float *__restrict__ weight,
                      const float *__restrict__ bias, const int32_t *__restrict__ cu,
                      const T *__restrict__ cache_in, T *__restrict__ y, int32_t N, int32_t T_,
                      int32_t C, int activation) {
    constexpr int V = Vec<T>::N;
    constexpr int R = kConvTB + W - 1;  // the block's rows and the W - 1 before them
    const int32_t c0 = (blockIdx.x * kConvThreads + threadIdx.x) * V;
    const int32_t t_begin = blockIdx.y * kConvTB;
    if (c0 >= C || t_begin >= T_) return;
    // every row this thread needs, as independent 16-byte loads issued up front
    typename Vec<T>::Raw raw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int32_t p = t_begin - (W - 1) + r;
        raw[r] = (p >= 0 && p < T_) ? Vec<T>::load_raw(x + (size_t)p * C + c0)
                                     : Vec<T>::zero_raw();
    }
    // the V channels' taps are V * W consecutive floats: vector loads
    float w[V][W], bsum[V];
    {
        const float *wp = weight + (size_t)c0 * W;
        if constexpr ((V * W) % 4 == 0) {
#pragma unroll
            for (int e = 0; e < V * W; e += 4) {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(wp + e));
                w[e / W][e % W] = f.x;
                w[(e + 1) / W][(e + 1) % W] = f.y;
                w[(e + 2) / W][(e + 2) % W] = f.z;
                w[(e + 3) / W][(e + 3) % W] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < V * W; ++e) w[e / W][e % W] = __ldg(wp + e);
        }
        if (bias) {
#pragma unroll
            for (int j = 0; j < V; j += 4) {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(bias + c0 + j));
                bsum[j] = f.x; bsum[j + 1] = f.y; bsum[j + 2] = f.z; bsum[j + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < V; ++j) bsum[j] = 0.f;
        }
    }
    // sequence bounds, clamped to [0, T) so bad offsets cannot address outside x
    int32_t s = seq_of(cu, N, t_begin);
    int32_t start = cu ? min(max(cu[s], 0), T_) : 0;
    int32_t next = cu ? min(max(cu[s + 1], start), T_) : T_;
    if (start <= t_begin - (W - 1) && next >= t_begin + kConvTB && t_begin + kConvTB <= T_) {
        // one sequence covers the block and its halo: a sliding window of
        // unpacked rows, no boundary tests
        float win[W][V];
#pragma unroll
        for (int r = 0; r < W - 1; ++r) Vec<T>::unpack(raw[r], win[r]);
#pragma unroll
        for (int jt = 0; jt < kConvTB; ++jt) {
            Vec<T>::unpack(raw[jt + W - 1], win[(jt + W - 1) % W]);
            float z[V];
#pragma unroll
            for (int j = 0; j < V; ++j) {
                float acc = bsum[j];
#pragma unroll
                for (int i = 0; i < W; ++i) acc = fmaf(w[j][i], win[(jt + i) % W][j], acc);
                z[j] = act(acc, activation);
            }
            Vec<T>::store(y + (size_t)(t_begin + jt) * C + c0, z);
        }
        return;
    }
#pragma unroll
    for (int jt = 0; jt < kConvTB; ++jt) {
        const int32_t t = t_begin + jt;
        if (t >= T_) break;
        while (t >= next && s + 1 < N) {  // a new sequence starts here (skipping empty ones)
            ++s;
            start = min(max(cu[s], 0), T_);
            next = min(max(cu[s + 1], start), T_);
        }
        float z[V];
#pragma unroll
        for (int j = 0; j < V; ++j) z[j] = bsum[j];
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const int32_t p = t - (W - 1) + i;
            float u[V];
            if (p >= start) {
                Vec<T>::unpack(raw[jt + i], u);
            } else if (cache_in) {
                // slot W - (start - p) of the sequence's cache, per channel
#pragma unroll
                for (int j = 0; j < V; ++j)
                    u[j] = (float)cache_in[((size_t)s * C + c0 + j) * W + W - (start - p)];
            } else {
#pragma unroll
                for (int j = 0; j < V; ++j) u[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < V; ++j) z[j] = fmaf(w[j][i], u[j], z[j]);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) z[j] = act(z[j], activation);
        Vec<T>::store(y + (size_t)t * C + c0, z);
    }
}

// cache_out[s, c, :] = the W most recent inputs of sequence s (its tokens,
// then what remains of cache_in when the sequence is shorter than W).  Each
// thread reads everything it writes first, so cache_out may be cache_in.
template <typename T, int W>
__global__ void short_conv_cache_kernel(const T *__restrict__ x, const int32_t *__restrict__ cu,
                                        const T *cache_in, T *cache_out, int32_t N, int32_t T_,
                                        int32_t C) {
    const int32_t c = blockIdx.x * blockDim.x + threadIdx.x, s = blockIdx.y;
    if (c >= C || s >= N) return;
    const int32_t a = cu ? min(max(cu[s], 0), T_) : 0;
    const int32_t b = cu ? min(max(cu[s + 1], a), T_) : T_;
    float v[W];
#pragma unroll
    for (int j = 0; j < W; ++j) {
        const int32_t p = b - W + j;
        if (p >= a) v[j] = (float)x[(size_t)p * C + c];
        else v[j] = cache_in ? (float)cache_in[((size_t)s * C + c) * W + W - (a - p)] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < W; ++j) cache_out[((size_t)s * C + c) * W + j] = (T)v[j];
}

// One decode token per sequence: shift the cache by one, append x, filter.
template <typename T, int W>
__global__ void short_conv_step_kernel(const T *__restrict__ x, const float *__restrict__ weight,
                                       const float *__restrict__ bias, T *cache,
                                       T *__restrict__ y, int32_t N, int32_t C, int activation) {
    const int32_t c = blockIdx.x * blockDim.x + threadIdx.x, n = blockIdx.y;
    if (c >= C || n >= N) return;
    T *cp = cache + ((size_t)n * C + c) * W;
    float win[W];
#pragma unroll
    for (int i = 0; i < W - 1; ++i) win[i] = (float)cp[i + 1];
    win[W - 1] = (float)x[(size_t)n * C + c];
    float z = bias ? bias[c] : 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) z = fmaf(weight[(size_t)c * W + i], win[i], z);
#pragma unroll
    for (int i = 0; i < W; ++i) cp[i] = (T)win[i];
    y[(size_t)n * C + c] = (T)act(z, activation);
}

template <typename T, int W>
cudaError_t launch_conv_t(const ConvArgs &a, cudaStream_t stream) {
    constexpr int V = Vec<T>::N;
    if (a.step) {
        const dim3 grid((unsigned)((a.C + 255) / 256), (unsigned)a.N);
        short_conv_step_kernel<T, W><<<grid, 256, 0, stream>>>(
            static_cast<const T *>(a.x), a.weight, a.bias, static_cast<T *>(a.cache_out),
            static_cast<T *>(a.y), a.N, a.C, a.activation);
        return cudaGetLastError();
    }
    if (a.T > 0) {
        const dim3 grid((unsigned)((a.C / V + kConvThreads - 1) / kConvThreads),
                        (unsigned)((a.T + kConvTB - 1) / kConvTB));
        short_conv_fwd_kernel<T, W><<<grid, kConvThreads, 0, stream>>>(
            static_cast<const T *>(a.x), a.weight, a.bias, a.cu_seqlens,
            static_cast<const T *>(a.cache_in), static_cast<T *>(a.y), a.N, a.T, a.C,
            a.activation);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.cache_out) {
        const dim3 grid((unsigned)((a.C + 255) / 256), (unsigned)a.N);
        short_conv_cache_kernel<T, W><<<grid, 256, 0, stream>>>(
            static_cast<const T *>(a.x), a.cu_seqlens, static_cast<const T *>(a.cache_in),
            static_cast<T *>(a.cache_out), a.N, a.T, a.C);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_dtype(const ConvArgs &a, cudaStream_t stream) {
    switch (a.W) {
        case 2: return launch_conv_t<T, 2>(a, stream);
        case 3: return launch_conv_t<T, 3>(a, stream);
        case 4: return launch_conv_t<T, 4>(a, stream);
        case 5: return launch_conv_t<T, 5>(a, stream);
        case 6: return launch_conv_t<T, 6>(a, stream);
        case 7: return launch_conv_t<T, 7>(a, stream);
        case 8: return launch_conv_t<T, 8>(a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_short_conv(const ConvArgs &a, cudaStream_t stream) {
    if (a.dtype == KDA_DTYPE_BF16) return launch_conv_dtype<__nv_bfloat16>(a, stream);
    return launch_conv_dtype<float>(a, stream);
}

}  // namespace kda
