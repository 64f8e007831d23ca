// fwd_recurrent.cu -- CUDA-core SSE forward, one CTA per segment, one token
// per step ("Scaling Linear Attention with Sparse State Expansion", eqs.
// 13-14 on the grouped per-partition subsequences of section 2.6, plus the
// always-on shared partition of section 2.5).
//
// Serves the float32 dtype (tight tolerance, no bf16 tensor-core operands)
// and any shape the tensor-core chunked path does not cover.  Each CTA walks
// its segment in time order with the c x d float32 state held in registers
// (thread = 4 columns x c/R rows) and writes, per token, the read-out of its
// partition as a float32 partial:
//   routed segment (b,h,i): part_routed[t,h,j,:] = e_t[i] * scale * q_t S_i
//   shared segment (b,h):   part_shared[t,h,:]   = scale * qs_t S_N
// The combine kernel sums the partials into out (the gated scatter-sum).
#include <algorithm>

#include "sse_internal.cuh"

namespace sse {
namespace {

constexpr int kRecThreads = 256;
constexpr int kRecMaxRows = 16;  // rows of the state per thread

template <typename T, int D4>
__global__ void __launch_bounds__(kRecThreads)
segment_recurrent_kernel(ForwardArgs a, int32_t H, int32_t c, int32_t N, int32_t topk,
                         int32_t use_shared, float scale) {
    constexpr int R = kRecThreads / D4;
    constexpr int d = 4 * D4;
    extern __shared__ float smem[];
    float *s_k = smem;        // [c]
    float *s_q = s_k + c;     // [c]
    float *s_a = s_q + c;     // [c]
    float *s_v = s_a + c;     // [d]
    float *s_red = s_v + d;   // [R][d]

    const T *q = static_cast<const T *>(a.q);
    const T *kk = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    const T *g = static_cast<const T *>(a.g);
    const T *qsb = static_cast<const T *>(a.qs ? a.qs : a.q);
    const T *ksb = static_cast<const T *>(a.ks ? a.ks : a.k);

    const int nshared = use_shared ? a.num_seqs * H : 0;
    const int P = N + use_shared;
    const bool is_shared = (int)blockIdx.x < nshared;
    int b, h, slot, len, base = 0;
    if (is_shared) {
        b = blockIdx.x / H;
        h = blockIdx.x % H;
        slot = N;
        base = a.cu_seqlens[b];
        len = a.cu_seqlens[b + 1] - base;
    } else {
        const int s = blockIdx.x - nshared;
        slot = s % N;
        h = (s / N) % H;
        b = s / (N * H);
        base = a.seg_off[s];
        len = a.seg_off[s + 1] - base;
    }
    const int cq = threadIdx.x % D4, rg = threadIdx.x / D4, col = 4 * cq;
    const int64_t state_off = (((int64_t)b * H + h) * P + slot) * (int64_t)c * d;

    float4 st[kRecMaxRows];
#pragma unroll
    for (int m = 0; m < kRecMaxRows; ++m) {
        const int r = rg + m * R;
        st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < c && a.init)
            st[m] = *reinterpret_cast<const float4 *>(a.init + state_off + (int64_t)r * d + col);
    }

    for (int n = 0; n < len; ++n) {
        int t, jj = 0;
        float e = 1.f;
        if (is_shared) {
            t = base + n;
        } else {
            const int rec = a.perm_rec[base + n];
            t = rec / topk;
            jj = rec - t * topk;
            e = a.topk_w[((int64_t)t * H + h) * topk + jj];
        }
        const int64_t th = (int64_t)t * H + h;
        const T *kr = (is_shared ? ksb : kk) + th * c;
        const T *qr = (is_shared ? qsb : q) + th * c;
        for (int r = threadIdx.x; r < c; r += kRecThreads) {
            s_k[r] = e * Elem<T>::load(kr + r);
            s_q[r] = e * scale * Elem<T>::load(qr + r);
            s_a[r] = expf(Elem<T>::load(g + th * c + r));
        }
        for (int cc = threadIdx.x; cc < d; cc += kRecThreads) s_v[cc] = Elem<T>::load(v + th * d + cc);
        __syncthreads();
        const float4 v4 = *reinterpret_cast<const float4 *>(s_v + col);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < kRecMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c) {
                const float ar = s_a[r], kr_ = s_k[r], qr_ = s_q[r];
                st[m].x = fmaf(ar, st[m].x, kr_ * v4.x);
                st[m].y = fmaf(ar, st[m].y, kr_ * v4.y);
                st[m].z = fmaf(ar, st[m].z, kr_ * v4.z);
                st[m].w = fmaf(ar, st[m].w, kr_ * v4.w);
                acc.x = fmaf(qr_, st[m].x, acc.x);
                acc.y = fmaf(qr_, st[m].y, acc.y);
                acc.z = fmaf(qr_, st[m].z, acc.z);
                acc.w = fmaf(qr_, st[m].w, acc.w);
            }
        }
        *reinterpret_cast<float4 *>(s_red + rg * d + col) = acc;
        __syncthreads();
        float *dst = is_shared ? static_cast<float *>(a.part_shared) + th * d
                               : static_cast<float *>(a.part_routed) + (th * topk + jj) * d;
        for (int cc = threadIdx.x; cc < d; cc += kRecThreads) {
            float o = 0.f;
            for (int r = 0; r < R; ++r) o += s_red[r * d + cc];
            dst[cc] = o;
        }
    }
    if (a.final_state) {
#pragma unroll
        for (int m = 0; m < kRecMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c)
                *reinterpret_cast<float4 *>(a.final_state + state_off + (int64_t)r * d + col) = st[m];
        }
    }
}

template <typename T, int D4>
cudaError_t launch_t(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    constexpr int R = kRecThreads / D4;
    const int c = cfg.key_dim, d = 4 * D4;
    const size_t smem = sizeof(float) * (3 * c + d + R * d);
    const int64_t nseg = (int64_t)a.num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    if (nseg == 0) return cudaSuccess;
    segment_recurrent_kernel<T, D4><<<(unsigned)nseg, kRecThreads, smem, stream>>>(
        a, cfg.num_heads, c, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_d(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    switch (cfg.value_dim) {
    case 16: return launch_t<T, 4>(cfg, a, stream);
    case 32: return launch_t<T, 8>(cfg, a, stream);
    case 64: return launch_t<T, 16>(cfg, a, stream);
    case 128: return launch_t<T, 32>(cfg, a, stream);
    case 256: return launch_t<T, 64>(cfg, a, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <typename P> struct PartLoad;
template <> struct PartLoad<float> {
    static __device__ __forceinline__ float4 load4(const float *p) {
        return *reinterpret_cast<const float4 *>(p);
    }
};
template <> struct PartLoad<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
};

// out[t,h,:] = sum_j part_routed[t,h,j,:] + part_shared[t,h,:], four columns per thread
template <typename T, typename P>
__global__ void combine_kernel(const P *__restrict__ part_routed, const P *__restrict__ part_shared,
                               int64_t rows, int32_t d, int32_t topk, T *__restrict__ out) {
    const int d4 = d / 4;
    const int64_t total = rows * d4;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = x / d4;
        const int col = (int)(x - row * d4) * 4;
        float4 o = part_shared ? PartLoad<P>::load4(part_shared + row * d + col) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < topk; ++j) {
            const float4 p = PartLoad<P>::load4(part_routed + (row * topk + j) * d + col);
            o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
        }
        Elem<T>::store4(out + row * d + col, o);
    }
}

template <typename T, typename P>
void launch_combine_t(const sse_config_t &cfg, const ForwardArgs &a, int64_t rows, unsigned blocks,
                      cudaStream_t stream) {
    const P *ps = cfg.use_shared ? static_cast<const P *>(a.part_shared) : nullptr;
    combine_kernel<T, P><<<blocks, 256, 0, stream>>>(static_cast<const P *>(a.part_routed), ps, rows,
                                                     cfg.value_dim, cfg.top_k, static_cast<T *>(a.out));
}

}  // namespace

bool recurrent_supported(const sse_config_t &cfg) {
    const int d = cfg.value_dim, c = cfg.key_dim;
    const bool d_ok = d == 16 || d == 32 || d == 64 || d == 128 || d == 256;
    if (!d_ok) return false;
    const int R = kRecThreads / (d / 4);
    return c >= 1 && c <= R * kRecMaxRows;
}

cudaError_t launch_forward_recurrent(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    if (cfg.dtype == SSE_BF16) return dispatch_d<__nv_bfloat16>(cfg, a, stream);
    return dispatch_d<float>(cfg, a, stream);
}

cudaError_t launch_combine(const sse_config_t &cfg, const ForwardArgs &a, cudaStream_t stream) {
    const int64_t rows = a.total_tokens * cfg.num_heads;
    if (rows == 0) return cudaSuccess;
    const int64_t work = rows * (cfg.value_dim / 4);
    const unsigned blocks = (unsigned)std::min<int64_t>((work + 255) / 256, 152 * 16);
    if (cfg.dtype == SSE_BF16) {
        if (a.part_bf16) launch_combine_t<__nv_bfloat16, __nv_bfloat16>(cfg, a, rows, blocks, stream);
        else launch_combine_t<__nv_bfloat16, float>(cfg, a, rows, blocks, stream);
    } else {
        if (a.part_bf16) launch_combine_t<float, __nv_bfloat16>(cfg, a, rows, blocks, stream);
        else launch_combine_t<float, float>(cfg, a, rows, blocks, stream);
    }
    return cudaGetLastError();
}

}  // namespace sse
