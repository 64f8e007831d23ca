// backward.cu -- gradients of the SSE layer ("Scaling Linear Attention with
// Sparse State Expansion", eqs. 9-14 and the shared partition of section 2.5)
// for L = <d_out, out> + <d_final_state, final_state>.
//
// Per (sequence, head, partition) segment -- the grouped subsequences of the
// varlen schedule (section 2.6), plus the shared partition over the whole
// sequence -- write the effective query and key of row t as
//   Q_t = w_t q_t   (w = e_t scale for a routed partition, scale for the shared one)
//   K_t = e_t k_t   (e = 1 for the shared one)
// so that S_t = diag(a_t) S_{t-1} + K_t^T v_t and o_t gets Q_t S_t.  One CTA
// per segment makes two sweeps, token by token in float32 on the CUDA cores:
//
//   forward : S_t from the initial state; u_t = S_t do_t^T (c);
//             dq_t = w_t u_t,  de_t(read) = scale q_t . u_t,  and Q_t * u_t
//             kept for the gate gradient;
//   reverse : dS = d_final_state (or 0); for t = last .. first:
//             dS += Q_t^T do_t;  dK_t = dS v_t^T (c);  dV_t = K_t dS (d);
//             dk_t = e_t dK_t,  dv_t = dV_t,  de_t(write) = k_t . dK_t;
//             dS <- diag(a_t) dS;
//             after the first row dS is the gradient of the initial state.
//
// The log-gate enters through G_t, the running sum of g over the segment's
// rows (S_t holds exp(G_t - G_s) K_s^T v_s and exp(G_t) S_0), so
//   dL/dG_t = Q_t * u_t - K_t * dK_t  (+ rowsum(S_T * dS_T) at the last row)
// and dL/dg_t is its reverse running sum over the segment -- no state before
// the step is needed.  Each segment writes its contribution of every row to a
// float32 slot [t, h, j] (j = the partition's place in the token's top-k,
// k for the shared one); a per-token kernel sums the slots in a fixed order
// and applies the router softmax's Jacobian over all N partitions:
//   dlogits = e * (de - <e, de>),  de zero at the unselected partitions
// (the top-k indices carry no gradient).
#include <algorithm>

#include "sse_internal.cuh"

namespace sse {
namespace {

constexpr int kBwdThreads = 256;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
constexpr int kBwdMaxRows = 16;  // state rows per thread

// Thread layout: D4 = d/4 column quads x R = 256/D4 row groups; thread
// (rg, cq) holds rows rg, rg + R, ... (at most kBwdMaxRows) x 4 columns of the
// state (forward sweep) and of its gradient (reverse sweep).
template <typename T, int D4>
__global__ void __launch_bounds__(kBwdThreads)
backward_segment_kernel(BackwardArgs a, int32_t H, int32_t c, int32_t N, int32_t topk, int32_t use_shared,
                        float scale) {
    constexpr int R = kBwdThreads / D4;
    constexpr int d = 4 * D4;
    extern __shared__ float smem[];
    // row inputs, double-buffered by row parity: [2][3c + 2d] = scale q, k,
    // exp(g), v, d_out
    const int row_floats = 3 * c + 2 * d;
    constexpr int D4P = D4 + 1;     // padded row stride: the per-row sums read conflict-free
    float *s_rows = smem + 2 * row_floats;  // [c][D4P] per-row partial sums over column quads
    float *s_cols = s_rows + c * D4P;       // [R][d] per-column partial sums over row groups
    float *s_red = s_cols + R * d;          // [2][kBwdThreads / 32] block reductions
    const T *q = static_cast<const T *>(a.q);
    const T *kk = static_cast<const T *>(a.k);
    const T *v = static_cast<const T *>(a.v);
    const T *g = static_cast<const T *>(a.g);
    const T *dout = static_cast<const T *>(a.d_out);
    const int ncon = topk + use_shared;
    const int nshared = use_shared ? a.num_seqs * H : 0;
    const int P = N + use_shared;
    // the work item: this CTA's index, or the list entry it names
    int item = (int)blockIdx.x;
    if (a.seg_list) {
        if (item >= *(volatile const int32_t *)a.seg_count) return;
        item = a.seg_list[item];
    }
    const bool is_shared = item < nshared;
    int b, h, slot, len, base;
    if (is_shared) {
        b = item / H;
        h = item % H;
        slot = N;
        base = a.cu_seqlens[b];
        len = a.cu_seqlens[b + 1] - base;
    } else {
        const int s = item - nshared;
        slot = s % N;
        h = (s / N) % H;
        b = s / (N * H);
        base = a.seg_off[s];
        len = a.seg_off[s + 1] - base;
    }
    const T *qsrc = is_shared && a.qs ? static_cast<const T *>(a.qs) : q;
    const T *ksrc = is_shared && a.ks ? static_cast<const T *>(a.ks) : kk;
    const int tid = threadIdx.x, cq = tid % D4, rg = tid / D4, col = 4 * cq;
    const int lane = tid & 31, warp = tid >> 5;
    const int64_t state_off = (((int64_t)b * H + h) * P + slot) * (int64_t)c * d;

    // row n of the segment: token, router weight e, contribution slot j
    auto row_info = [&](int n, int &t, float &e, int &j) {
        if (is_shared) {
            t = base + n;
            e = 1.f;
            j = topk;
        } else {
            const int rec = a.perm_rec[base + n];
            t = rec / topk;
            j = rec - t * topk;
            e = a.perm_e[base + n];
        }
    };
    // Row inputs travel in two steps: the next row's values are loaded into
    // registers (one element of each tensor per thread: c, d <= 256) while
    // the current row computes, then stored into the other shared buffer.
    // The registers hold the raw elements: any arithmetic on a loaded value
    // would make the warp wait for the load right here.
    struct RowRegs { T q, k, g, v, d; };
    auto fetch_row = [&](int t) -> RowRegs {
        RowRegs x{};
        const int64_t th = (int64_t)t * H + h;
        if (tid < c) {
            x.q = qsrc[th * c + tid];
            x.k = ksrc[th * c + tid];
            x.g = g[th * c + tid];
        }
        if (tid < d) {
            x.v = v[th * d + tid];
            x.d = dout[th * d + tid];
        }
        return x;
    };
    auto store_row = [&](const RowRegs &x, float *buf) {
        if (tid < c) {
            buf[tid] = scale * to_f32(x.q);
            buf[c + tid] = to_f32(x.k);
            buf[2 * c + tid] = expf(to_f32(x.g));
        }
        if (tid < d) {
            buf[3 * c + tid] = to_f32(x.v);
            buf[3 * c + d + tid] = to_f32(x.d);
        }
    };
    // block-wide sum of one float per thread (every thread gets the result);
    // its two halves of s_red alternate by call parity, so one barrier suffices
    int red_parity = 0;
    auto block_sum = [&](float x) -> float {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        float *red = s_red + red_parity * (kBwdThreads / 32);
        red_parity ^= 1;
        if (lane == 0) red[warp] = x;
        __syncthreads();
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kBwdThreads / 32; ++w) s += red[w];
        return s;
    };

    float4 st[kBwdMaxRows];
#pragma unroll
    for (int m = 0; m < kBwdMaxRows; ++m) {
        const int r = rg + m * R;
        st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < c && a.init)
            st[m] = *reinterpret_cast<const float4 *>(a.init + state_off + (int64_t)r * d + col);
    }

    // ---- forward sweep: S_t, u_t = S_t do_t^T ---------------------------------
    int t_next = 0, j_next = 0;
    float e_next = 0.f;
    RowRegs x_next{};
    if (len > 0) {
        row_info(0, t_next, e_next, j_next);
        x_next = fetch_row(t_next);
    }
    for (int n = 0; n < len; ++n) {
        const int t = t_next, j = j_next;
        const float e = e_next;
        float *buf = smem + (n & 1) * row_floats;
        store_row(x_next, buf);
        if (n + 1 < len) {  // the next row's inputs load while this row computes
            row_info(n + 1, t_next, e_next, j_next);
            x_next = fetch_row(t_next);
        }
        __syncthreads();
        const float *s_q = buf, *s_k = buf + c, *s_a = buf + 2 * c, *s_v = buf + 3 * c, *s_do = s_v + d;
        const float4 v4 = *reinterpret_cast<const float4 *>(s_v + col);
        const float4 d4 = *reinterpret_cast<const float4 *>(s_do + col);
#pragma unroll
        for (int m = 0; m < kBwdMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c) {
                const float ar = s_a[r], kr = e * s_k[r];
                st[m].x = fmaf(ar, st[m].x, kr * v4.x);
                st[m].y = fmaf(ar, st[m].y, kr * v4.y);
                st[m].z = fmaf(ar, st[m].z, kr * v4.z);
                st[m].w = fmaf(ar, st[m].w, kr * v4.w);
                s_rows[r * D4P + cq] = st[m].x * d4.x + st[m].y * d4.y + st[m].z * d4.z + st[m].w * d4.w;
            }
        }
        __syncthreads();
        float qu = 0.f;
        const int64_t slot_row = ((int64_t)t * H + h) * ncon + j;
        if (tid < c) {
            float u = 0.f;
            for (int x = 0; x < D4; ++x) u += s_rows[tid * D4P + x];
            Elem<T>::store(static_cast<T *>(a.dq_c) + slot_row * c + tid, e * scale * u);
            a.dg_c[slot_row * c + tid] = e * s_q[tid] * u;  // Q * u, finished by the reverse sweep
            qu = s_q[tid] * u;
        }
        // its barrier also orders this row's reads of s_rows before the next row's writes
        const float de_read = block_sum(qu);
        if (!is_shared && tid == 0) a.de_c[(((int64_t)t * H + h) * topk + j) * 2] = de_read;
    }

    // ---- reverse sweep: dS, dK, dV, gate gradient -----------------------------
    // gradient of the final state, and its term rowsum(S_T * dS_T) of dL/dG
    float4 ds[kBwdMaxRows];
#pragma unroll
    for (int m = 0; m < kBwdMaxRows; ++m) {
        const int r = rg + m * R;
        ds[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < c && a.d_final)
            ds[m] = *reinterpret_cast<const float4 *>(a.d_final + state_off + (int64_t)r * d + col);
        if (r < c)
            s_rows[r * D4P + cq] = st[m].x * ds[m].x + st[m].y * ds[m].y + st[m].z * ds[m].z + st[m].w * ds[m].w;
    }
    __syncthreads();
    float run = 0.f;  // reverse running sum of dL/dG for row tid (tid < c)
    if (tid < c)
        for (int x = 0; x < D4; ++x) run += s_rows[tid * D4P + x];
    __syncthreads();
    // Q * u of the row (from the forward sweep) travels with the row's inputs
    auto fetch_qu = [&](int t, int j) -> float {
        return tid < c ? a.dg_c[(((int64_t)t * H + h) * ncon + j) * c + tid] : 0.f;
    };
    float qu_next = 0.f;
    if (len > 0) {
        row_info(len - 1, t_next, e_next, j_next);
        x_next = fetch_row(t_next);
        qu_next = fetch_qu(t_next, j_next);
    }
    for (int n = len - 1; n >= 0; --n) {
        const int t = t_next, j = j_next;
        const float e = e_next, qu_row = qu_next;
        float *buf = smem + (n & 1) * row_floats;
        store_row(x_next, buf);
        if (n > 0) {
            row_info(n - 1, t_next, e_next, j_next);
            x_next = fetch_row(t_next);
            qu_next = fetch_qu(t_next, j_next);
        }
        __syncthreads();
        const float *s_q = buf, *s_k = buf + c, *s_a = buf + 2 * c, *s_v = buf + 3 * c, *s_do = s_v + d;
        const float4 v4 = *reinterpret_cast<const float4 *>(s_v + col);
        const float4 d4 = *reinterpret_cast<const float4 *>(s_do + col);
        float4 dv_part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < kBwdMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c) {
                const float qr = e * s_q[r], kr = e * s_k[r];
                ds[m].x = fmaf(qr, d4.x, ds[m].x);
                ds[m].y = fmaf(qr, d4.y, ds[m].y);
                ds[m].z = fmaf(qr, d4.z, ds[m].z);
                ds[m].w = fmaf(qr, d4.w, ds[m].w);
                s_rows[r * D4P + cq] = ds[m].x * v4.x + ds[m].y * v4.y + ds[m].z * v4.z + ds[m].w * v4.w;
                dv_part.x = fmaf(kr, ds[m].x, dv_part.x);
                dv_part.y = fmaf(kr, ds[m].y, dv_part.y);
                dv_part.z = fmaf(kr, ds[m].z, dv_part.z);
                dv_part.w = fmaf(kr, ds[m].w, dv_part.w);
                const float ar = s_a[r];
                ds[m].x *= ar;
                ds[m].y *= ar;
                ds[m].z *= ar;
                ds[m].w *= ar;
            }
        }
        *reinterpret_cast<float4 *>(s_cols + rg * d + col) = dv_part;
        __syncthreads();
        const int64_t slot_row = ((int64_t)t * H + h) * ncon + j;
        float kdk = 0.f;
        if (tid < c) {
            float dkr = 0.f;
            for (int x = 0; x < D4; ++x) dkr += s_rows[tid * D4P + x];
            Elem<T>::store(static_cast<T *>(a.dk_c) + slot_row * c + tid, e * dkr);
            kdk = s_k[tid] * dkr;
            // dL/dG_t = Q_t * u_t - K_t * dK_t, summed from the last row down
            run += qu_row - e * kdk;
            a.dg_c[slot_row * c + tid] = run;
        }
        for (int cc = tid; cc < d; cc += kBwdThreads) {
            float s = 0.f;
            for (int r2 = 0; r2 < R; ++r2) s += s_cols[r2 * d + cc];
            Elem<T>::store(static_cast<T *>(a.dv_c) + slot_row * d + cc, s);
        }
        // its barrier also orders this row's reads of s_rows / s_cols before the next row's writes
        const float de_write = block_sum(kdk);
        if (!is_shared && tid == 0) a.de_c[(((int64_t)t * H + h) * topk + j) * 2 + 1] = de_write;
    }
    if (a.d_init) {
#pragma unroll
        for (int m = 0; m < kBwdMaxRows; ++m) {
            const int r = rg + m * R;
            if (r < c) *reinterpret_cast<float4 *>(a.d_init + state_off + (int64_t)r * d + col) = ds[m];
        }
    }
}

// G consecutive elements (G = 4: 8-byte bf16 / 16-byte float accesses; G = 8:
// 16-byte bf16 / two 16-byte float accesses) as float32.
template <typename T, int G> struct Cols;
template <typename T> struct Cols<T, 4> {
    static __device__ __forceinline__ void load(const T *p, float (&x)[4]) {
        const float4 y = Elem<T>::load4(p);
        x[0] = y.x; x[1] = y.y; x[2] = y.z; x[3] = y.w;
    }
    static __device__ __forceinline__ void store(T *p, const float (&x)[4]) {
        Elem<T>::store4(p, make_float4(x[0], x[1], x[2], x[3]));
    }
};
template <typename T> struct Cols<T, 8> {
    static __device__ __forceinline__ void load(const T *p, float (&x)[8]) {
        if constexpr (sizeof(T) == 2) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[2 * i] = __uint_as_float(w[i] << 16);
                x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        } else {
            const float4 y0 = Elem<T>::load4(p), y1 = Elem<T>::load4(p + 4);
            x[0] = y0.x; x[1] = y0.y; x[2] = y0.z; x[3] = y0.w;
            x[4] = y1.x; x[5] = y1.y; x[6] = y1.z; x[7] = y1.w;
        }
    }
    static __device__ __forceinline__ void store(T *p, const float (&x)[8]) {
        if constexpr (sizeof(T) == 2) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            Elem<T>::store4(p, make_float4(x[0], x[1], x[2], x[3]));
            Elem<T>::store4(p + 4, make_float4(x[4], x[5], x[6], x[7]));
        }
    }
};
template <int G>
__device__ __forceinline__ void load_f32(const float *p, float (&x)[G]) {
#pragma unroll
    for (int i = 0; i < G; i += 4) {
        const float4 y = *reinterpret_cast<const float4 *>(p + i);
        x[i] = y.x; x[i + 1] = y.y; x[i + 2] = y.z; x[i + 3] = y.w;
    }
}

// Per (t, h): the fixed-order sums of the contribution slots, and the router
// logits' gradient through the softmax over all N partitions.  One thread per
// (t, h) row handles its logits; then the c- and d-wide sums run G columns
// per thread, NC (= k + shared) slot loads issued before the sum.
template <typename T, int NC, int G>
__global__ void __launch_bounds__(256)
backward_combine_kernel(BackwardArgs a, int64_t rows, int32_t c, int32_t d, int32_t N, int32_t topk,
                        int32_t use_shared) {
    const int ncon = NC;
    const int cg = c / G, dg = d / G;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t gid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    const bool sep_q = use_shared && a.qs, sep_k = use_shared && a.ks;
    for (int64_t row = gid; row < rows; row += stride) {
        // dlogits = e * (de - <e, de>): softmax of the stored logits in fp32
        const T *lg = static_cast<const T *>(a.logits) + row * N;
        float m = -INFINITY;
        for (int i = 0; i < N; ++i) m = fmaxf(m, Elem<T>::load(lg + i));
        float s = 0.f;
        for (int i = 0; i < N; ++i) s += expf(Elem<T>::load(lg + i) - m);
        const float inv = 1.f / s;
        float ede = 0.f;
        for (int j = 0; j < topk; ++j) {
            const int i = a.topk_idx[row * topk + j];
            ede += expf(Elem<T>::load(lg + i) - m) * inv * (a.de_c[(row * topk + j) * 2] + a.de_c[(row * topk + j) * 2 + 1]);
        }
        T *dl = static_cast<T *>(a.d_logits) + row * N;
        for (int i = 0; i < N; ++i) {
            float de = 0.f;
            for (int j = 0; j < topk; ++j)
                if (a.topk_idx[row * topk + j] == i) de = a.de_c[(row * topk + j) * 2] + a.de_c[(row * topk + j) * 2 + 1];
            const float e = expf(Elem<T>::load(lg + i) - m) * inv;
            Elem<T>::store(dl + i, e * (de - ede));
        }
    }
    const int per_row = 4 * cg + dg;  // dq, dk, dg, dq_shared / dk_shared, dv
    const int64_t total = rows * per_row;
    const T *sq = static_cast<const T *>(a.dq_c), *sk = static_cast<const T *>(a.dk_c);
    const T *sv = static_cast<const T *>(a.dv_c);
    // (row, part) of element x: 32-bit unsigned division when every index fits,
    // a 64-bit one (emulated, several times slower) otherwise
    const bool idx32 = total <= (int64_t)0xffffffffu;
    for (int64_t x = gid; x < total; x += stride) {
        int64_t row;
        uint32_t part;
        if (idx32) {
            const uint32_t xr = (uint32_t)x, r32 = xr / (uint32_t)per_row;
            row = r32;
            part = xr - r32 * (uint32_t)per_row;
        } else {
            row = x / per_row;
            part = (uint32_t)(x - row * per_row);
        }
        const T *src = nullptr;  // dq, dk, dv slots (I/O type); dg slots are float32
        T *dst;
        int width, cidx, hi;  // slots 0 .. hi - 1 summed
        const uint32_t ucg = (uint32_t)cg;
        const int kind = part < 4 * ucg ? (int)(part / ucg) : 4;
        if (kind < 4) {
            cidx = G * (int)(part % ucg);
            width = c;
            // 0: dq (routed slots, plus the shared slot unless q_shared is separate),
            // 1: dk (likewise), 2: dg (all slots), 3: dq_shared / dk_shared
            if (kind == 0) { src = sq; dst = static_cast<T *>(a.dq); hi = sep_q ? topk : ncon; }
            else if (kind == 1) { src = sk; dst = static_cast<T *>(a.dk); hi = sep_k ? topk : ncon; }
            else if (kind == 2) { dst = static_cast<T *>(a.dg); hi = ncon; }
            else {
                // the shared slot alone, into dq_shared and dk_shared when they are separate
                float y[G];
                if (sep_q) {
                    Cols<T, G>::load(sq + (row * ncon + topk) * c + cidx, y);
                    Cols<T, G>::store(static_cast<T *>(a.dq_shared) + row * c + cidx, y);
                }
                if (sep_k) {
                    Cols<T, G>::load(sk + (row * ncon + topk) * c + cidx, y);
                    Cols<T, G>::store(static_cast<T *>(a.dk_shared) + row * c + cidx, y);
                }
                continue;
            }
        } else {
            cidx = G * (int)(part - 4 * ucg);
            width = d;
            src = sv;
            dst = static_cast<T *>(a.dv);
            hi = ncon;
        }
        float p[NC][G];
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const int64_t o = (row * ncon + j) * width + cidx;
            if (j >= hi) {
#pragma unroll
                for (int i = 0; i < G; ++i) p[j][i] = 0.f;
            } else if (src) {
                Cols<T, G>::load(src + o, p[j]);
            } else {
                load_f32<G>(a.dg_c + o, p[j]);
            }
        }
        float acc[G];
#pragma unroll
        for (int i = 0; i < G; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            if (j >= hi) break;
#pragma unroll
            for (int i = 0; i < G; ++i) acc[i] += p[j][i];
        }
        Cols<T, G>::store(dst + row * width + cidx, acc);
    }
}

template <typename T, int D4>
cudaError_t launch_segments(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream) {
    constexpr int R = kBwdThreads / D4;
    const int c = cfg.key_dim, d = 4 * D4;
    const size_t smem = sizeof(float) * (2 * (3 * c + 2 * d) + c * (D4 + 1) + R * d + 2 * (kBwdThreads / 32));
    const int64_t nseg = (int64_t)a.num_seqs * cfg.num_heads * (cfg.num_partitions + cfg.use_shared);
    if (nseg == 0) return cudaSuccess;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(backward_segment_kernel<T, D4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    backward_segment_kernel<T, D4><<<(unsigned)nseg, kBwdThreads, smem, stream>>>(
        a, cfg.num_heads, c, cfg.num_partitions, cfg.top_k, cfg.use_shared, cfg.scale);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_d(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream) {
    switch (cfg.value_dim) {
    case 16: return launch_segments<T, 4>(cfg, a, stream);
    case 32: return launch_segments<T, 8>(cfg, a, stream);
    case 64: return launch_segments<T, 16>(cfg, a, stream);
    case 128: return launch_segments<T, 32>(cfg, a, stream);
    case 256: return launch_segments<T, 64>(cfg, a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_backward_segments(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream) {
    return cfg.dtype == SSE_BF16 ? dispatch_d<__nv_bfloat16>(cfg, a, stream) : dispatch_d<float>(cfg, a, stream);
}

// Eight columns per thread where every row and output is 16-byte aligned,
// four otherwise.
template <typename T, int G>
cudaError_t launch_combine_g(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream) {
    const int64_t rows = a.total_tokens * cfg.num_heads;
    const int per_row = 4 * (cfg.key_dim / G) + cfg.value_dim / G;
    const unsigned blocks = (unsigned)std::min<int64_t>((rows * per_row + 255) / 256, 152 * 16);
#define SSE_BCOMB(NC)                                                                                         \
    case NC:                                                                                                  \
        backward_combine_kernel<T, NC, G><<<blocks, 256, 0, stream>>>(a, rows, cfg.key_dim, cfg.value_dim,  \
                                                                      cfg.num_partitions, cfg.top_k,          \
                                                                      cfg.use_shared);                        \
        break
    switch (cfg.top_k + cfg.use_shared) {
        SSE_BCOMB(1); SSE_BCOMB(2); SSE_BCOMB(3); SSE_BCOMB(4); SSE_BCOMB(5);
        SSE_BCOMB(6); SSE_BCOMB(7); SSE_BCOMB(8); SSE_BCOMB(9);
        default: return cudaErrorInvalidValue;
    }
#undef SSE_BCOMB
    return cudaGetLastError();
}

cudaError_t launch_backward_combine(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream) {
    const int64_t rows = a.total_tokens * cfg.num_heads;
    if (rows == 0) return cudaSuccess;
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool g8 = cfg.key_dim % 8 == 0 && cfg.value_dim % 8 == 0 && al16(a.dq) && al16(a.dk) && al16(a.dv) &&
                    al16(a.dg) && (!a.dq_shared || al16(a.dq_shared)) && (!a.dk_shared || al16(a.dk_shared));
    if (cfg.dtype == SSE_BF16)
        return g8 ? launch_combine_g<__nv_bfloat16, 8>(cfg, a, stream) : launch_combine_g<__nv_bfloat16, 4>(cfg, a, stream);
    return g8 ? launch_combine_g<float, 8>(cfg, a, stream) : launch_combine_g<float, 4>(cfg, a, stream);
}

bool backward_supported(const sse_config_t &cfg) {
    const int d = cfg.value_dim, c = cfg.key_dim;
    if (!(d == 16 || d == 32 || d == 64 || d == 128 || d == 256)) return false;
    const int R = kBwdThreads / (d / 4);
    return c >= 4 && c % 4 == 0 && c <= R * kBwdMaxRows && c <= kBwdThreads;
}

cudaError_t launch_backward(const sse_config_t &cfg, const BackwardArgs &a, cudaStream_t stream, int *launches) {
    cudaError_t e = launch_backward_segments(cfg, a, stream);
    if (e != cudaSuccess) return e;
    *launches += 1;
    e = launch_backward_combine(cfg, a, stream);
    *launches += 1;
    return e;
}

}  // namespace sse
