// decode.cu -- one SSE decode step on states resident in HBM ("Scaling
// Linear Attention with Sparse State Expansion", section 2.6: decoding recurs
// only on the selected states; update and read-out of eqs. 13-14 and the
// shared partition of section 2.5).
//
// One CTA per (sequence, head).  Warp 0 routes the token (softmax + top-k
// over N logits, by shuffles); the token vectors go to shared memory; then the CTA streams
// exactly k + use_shared states (c x d float32 each) through registers:
//   S <- diag(exp g) S + w_write k^T v   (read-modify-write, 16-byte vectors)
//   o += w_read q S                      (partial per thread, reduced in smem)
// Thread layout: D4 = d/4 column quads per row; a warp covers whole rows, so
// every load/store instruction of a warp touches contiguous 512-byte rows.
// Unselected states are never read or written.
#include "sse_internal.cuh"

namespace sse {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kBatch = 8;  // state rows per thread in flight

template <typename T, int D4>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(const T *__restrict__ q, const T *__restrict__ kk, const T *__restrict__ v,
              const T *__restrict__ g, const T *__restrict__ logits, const T *__restrict__ qs,
              const T *__restrict__ ks, int32_t H, int32_t c, int32_t N, int32_t topk,
              int32_t use_shared, float scale, float *__restrict__ state, T *__restrict__ out,
              int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
    constexpr int R = kDecodeThreads / D4;  // row groups
    constexpr int d = 4 * D4;
    extern __shared__ float smem[];
    float *s_a = smem;         // [c]   exp(g)
    float *s_k = s_a + c;      // [c]
    float *s_q = s_k + c;      // [c]
    float *s_ks = s_q + c;     // [c]
    float *s_qs = s_ks + c;    // [c]
    float *s_v = s_qs + c;     // [d]
    float *s_red = s_v + d;    // [R][d]
    __shared__ int s_slot[kMaxTopK + 1];
    __shared__ float s_ww[kMaxTopK + 1], s_wr[kMaxTopK + 1];

    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    const T *qrow = q + bh * c, *krow = kk + bh * c, *grow = g + bh * c;
    const T *qsrow = (qs ? qs : q) + bh * c, *ksrow = (ks ? ks : kk) + bh * c;
    for (int r = tid; r < c; r += kDecodeThreads) {
        s_a[r] = expf(Elem<T>::load(grow + r));
        s_k[r] = Elem<T>::load(krow + r);
        s_q[r] = Elem<T>::load(qrow + r);
        s_ks[r] = Elem<T>::load(ksrow + r);
        s_qs[r] = Elem<T>::load(qsrow + r);
    }
    for (int col = tid; col < d; col += kDecodeThreads) s_v[col] = Elem<T>::load(v + bh * d + col);
    if (tid < 32) {  // warp 0 routes the token
        int idx[kMaxTopK];
        float w[kMaxTopK];
        route_token_warp<T>(logits + bh * N, N, topk, tid, idx, w);
        for (int j = 0; j < topk && tid == 0; ++j) {
            s_slot[j] = idx[j];
            s_ww[j] = w[j];
            s_wr[j] = w[j] * scale;
            if (topk_idx) topk_idx[bh * topk + j] = idx[j];
            if (topk_w) topk_w[bh * topk + j] = w[j];
        }
        if (use_shared && tid == 0) {
            s_slot[topk] = N;
            s_ww[topk] = 1.f;
            s_wr[topk] = scale;
        }
    }
    __syncthreads();

    const int P = N + use_shared;
    const int nslots = topk + use_shared;
    const int cq = tid % D4;   // column quad
    const int rg = tid / D4;   // row group
    const int col = 4 * cq;
    const float4 v4 = make_float4(s_v[col], s_v[col + 1], s_v[col + 2], s_v[col + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sl = 0; sl < nslots; ++sl) {
        const bool shared_slot = use_shared && sl == topk;
        const float *kvec = shared_slot ? s_ks : s_k;
        const float *qvec = shared_slot ? s_qs : s_q;
        const float ww = s_ww[sl], wr = s_wr[sl];
        float *S = state + (bh * P + s_slot[sl]) * (int64_t)c * d;
        // kBatch rows per thread in flight: all loads of a batch are issued
        // before its first store
        for (int r0 = rg; r0 < c; r0 += kBatch * R) {
            float4 sv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int r = r0 + u * R;
                if (r < c) sv[u] = __ldcs(reinterpret_cast<const float4 *>(S + (int64_t)r * d + col));
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int r = r0 + u * R;
                if (r < c) {
                    float4 s = sv[u];
                    const float a = s_a[r], kw = ww * kvec[r], qw = wr * qvec[r];
                    s.x = fmaf(a, s.x, kw * v4.x);
                    s.y = fmaf(a, s.y, kw * v4.y);
                    s.z = fmaf(a, s.z, kw * v4.z);
                    s.w = fmaf(a, s.w, kw * v4.w);
                    __stcs(reinterpret_cast<float4 *>(S + (int64_t)r * d + col), s);
                    acc.x = fmaf(qw, s.x, acc.x);
                    acc.y = fmaf(qw, s.y, acc.y);
                    acc.z = fmaf(qw, s.z, acc.z);
                    acc.w = fmaf(qw, s.w, acc.w);
                }
            }
        }
    }
    *reinterpret_cast<float4 *>(s_red + rg * d + col) = acc;
    __syncthreads();
    for (int cc = tid; cc < d; cc += kDecodeThreads) {
        float o = 0.f;
#pragma unroll 8
        for (int r = 0; r < R; ++r) o += s_red[r * d + cc];
        Elem<T>::store(out + bh * d + cc, o);
    }
}

template <typename T, int D4>
cudaError_t launch_t(const sse_config_t &cfg, const void *q, const void *k, const void *v,
                     const void *g, const void *logits, const void *qs, const void *ks,
                     int32_t batch, float *state, void *out, int32_t *topk_idx, float *topk_w,
                     cudaStream_t stream) {
    constexpr int R = kDecodeThreads / D4;
    const int c = cfg.key_dim, d = 4 * D4;
    const size_t smem = sizeof(float) * (5 * c + d + R * d);
    const int64_t blocks = (int64_t)batch * cfg.num_heads;
    decode_kernel<T, D4><<<(unsigned)blocks, kDecodeThreads, smem, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<const T *>(g), static_cast<const T *>(logits), static_cast<const T *>(qs),
        static_cast<const T *>(ks), cfg.num_heads, c, cfg.num_partitions, cfg.top_k,
        cfg.use_shared, cfg.scale, state, static_cast<T *>(out), topk_idx, topk_w);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_d(const sse_config_t &cfg, const void *q, const void *k, const void *v,
                       const void *g, const void *logits, const void *qs, const void *ks,
                       int32_t batch, float *state, void *out, int32_t *topk_idx, float *topk_w,
                       cudaStream_t stream) {
    switch (cfg.value_dim) {
    case 16: return launch_t<T, 4>(cfg, q, k, v, g, logits, qs, ks, batch, state, out, topk_idx, topk_w, stream);
    case 32: return launch_t<T, 8>(cfg, q, k, v, g, logits, qs, ks, batch, state, out, topk_idx, topk_w, stream);
    case 64: return launch_t<T, 16>(cfg, q, k, v, g, logits, qs, ks, batch, state, out, topk_idx, topk_w, stream);
    case 128: return launch_t<T, 32>(cfg, q, k, v, g, logits, qs, ks, batch, state, out, topk_idx, topk_w, stream);
    case 256: return launch_t<T, 64>(cfg, q, k, v, g, logits, qs, ks, batch, state, out, topk_idx, topk_w, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_supported(const sse_config_t &cfg) {
    const int d = cfg.value_dim, c = cfg.key_dim;
    const bool d_ok = d == 16 || d == 32 || d == 64 || d == 128 || d == 256;
    return d_ok && c >= 1 && c <= 1024;
}

cudaError_t launch_decode(const sse_config_t &cfg, const void *q, const void *k, const void *v,
                          const void *g, const void *logits, const void *qs, const void *ks,
                          int32_t batch, float *state, void *out, int32_t *topk_idx,
                          float *topk_w, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    if (cfg.dtype == SSE_BF16)
        return dispatch_d<__nv_bfloat16>(cfg, q, k, v, g, logits, qs, ks, batch, state, out,
                                         topk_idx, topk_w, stream);
    return dispatch_d<float>(cfg, q, k, v, g, logits, qs, ks, batch, state, out, topk_idx,
                             topk_w, stream);
}

}  // namespace sse
