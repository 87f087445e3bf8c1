// Memory-bound helpers around the ring fold:
//  * merge  -- fold one partial attention result (O_b, lse_b) over a disjoint
//              key set into another (O_a, lse_a): the log-sum-exp weighted
//              rescale-and-add that the online softmax performs when a new
//              block arrives (aiunderstanding.org, "Approfondimento
//              tecnico"; glossary page, running-max remark).
//  * relayout -- bit-exact row permutation between token order and a
//              shard-major layout: striped, token t <-> row (t mod N)*Sb +
//              t div N (glossary page, Striped Attention), or zigzag, shard i
//              holding chunks i and 2N-1-i of 2N chunks (the Zulu
//              aiunderstanding.org page names the variant; this layout is the
//              build's reading of it).
//  * ulysses -- the all-to-all of DeepSpeed Ulysses (glossary page, comparison
//              with other kinds of parallelism) as a permutation between N
//              device-contiguous buffers: sequence-sharded <-> head-sharded.
// Rows of 2..32 16-byte vectors use the row-group kernels (several rows per
// warp, every lane moving 16 bytes, loads batched ahead of stores); other
// shapes fall back to one warp per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ra.h"

namespace ra {
namespace aux {

constexpr int kBlock = 256;

template <typename T>
struct Vec;  // 16-byte vector of T
template <>
struct Vec<float> {
    static constexpr int n = 4;
    __device__ static void fma2(uint4& a, const uint4& b, float ca, float cb) {
        a.x = __float_as_uint(ca * __uint_as_float(a.x) + cb * __uint_as_float(b.x));
        a.y = __float_as_uint(ca * __uint_as_float(a.y) + cb * __uint_as_float(b.y));
        a.z = __float_as_uint(ca * __uint_as_float(a.z) + cb * __uint_as_float(b.z));
        a.w = __float_as_uint(ca * __uint_as_float(a.w) + cb * __uint_as_float(b.w));
    }
};
__device__ __forceinline__ uint32_t mix_bf16x2(uint32_t a, uint32_t b, float ca, float cb) {
    __nv_bfloat162 va = *reinterpret_cast<__nv_bfloat162*>(&a);
    __nv_bfloat162 vb = *reinterpret_cast<__nv_bfloat162*>(&b);
    float2 fa = __bfloat1622float2(va), fb = __bfloat1622float2(vb);
    __nv_bfloat162 r = __floats2bfloat162_rn(ca * fa.x + cb * fb.x, ca * fa.y + cb * fb.y);
    return *reinterpret_cast<uint32_t*>(&r);
}
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void fma2(uint4& a, const uint4& b, float ca, float cb) {
        a.x = mix_bf16x2(a.x, b.x, ca, cb);
        a.y = mix_bf16x2(a.y, b.y, ca, cb);
        a.z = mix_bf16x2(a.z, b.z, ca, cb);
        a.w = mix_bf16x2(a.w, b.w, ca, cb);
    }
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float x) { d = __float2bfloat16_rn(x); }

template <typename T, bool VEC>
__global__ void __launch_bounds__(kBlock) merge_kernel(T* __restrict__ oa, float* __restrict__ la,
                                                       const T* __restrict__ ob,
                                                       const float* __restrict__ lb, int64_t rows,
                                                       int D) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kBlock / 32);
    for (int64_t row = (int64_t)blockIdx.x * (kBlock / 32) + threadIdx.x / 32; row < rows;
         row += warps) {
        const float a = la[row], b = lb[row];
        const float mx = fmaxf(a, b);
        float ca = 0.f, cb = 0.f, lse = -INFINITY;
        if (mx != -INFINITY) {
            const float wa = expf(a - mx), wb = expf(b - mx);  // exp(-inf) = 0
            const float tot = wa + wb;
            lse = mx + logf(tot);
            ca = wa / tot;
            cb = wb / tot;
        }
        T* ra_ = oa + row * D;
        const T* rb = ob + row * D;
        if (VEC) {
            constexpr int n = Vec<T>::n;
            uint4* va = reinterpret_cast<uint4*>(ra_);
            const uint4* vb = reinterpret_cast<const uint4*>(rb);
            for (int e = lane; e < D / n; e += 32) {
                uint4 x = va[e];
                const uint4 y = vb[e];
                Vec<T>::fma2(x, y, ca, cb);
                va[e] = x;
            }
        } else {
            for (int e = lane; e < D; e += 32) from_f(ra_[e], ca * to_f(ra_[e]) + cb * to_f(rb[e]));
        }
        __syncwarp();
        if (lane == 0) la[row] = lse;
    }
}

// Shard-major row of token t (layout 1 striped, 2 zigzag, else contiguous).
__device__ __forceinline__ int64_t row_of_token(int64_t t, int64_t Sb, int64_t N, int layout) {
    if (layout == 1) return (t % N) * Sb + t / N;
    if (layout == 2) {
        const int64_t h = Sb / 2, c = t / h, o = t % h;
        return c < N ? c * Sb + o : (2 * N - 1 - c) * Sb + h + o;
    }
    return t;
}
// Token held by shard-major row p.
__device__ __forceinline__ int64_t token_of_row(int64_t p, int64_t Sb, int64_t N, int layout) {
    const int64_t i = p / Sb, r = p % Sb;
    if (layout == 1) return r * N + i;
    if (layout == 2) {
        const int64_t h = Sb / 2;
        return r < h ? i * h + r : (2 * N - 1 - i) * h + (r - h);
    }
    return p;
}
// Source row (within a slice) of destination row p.
__device__ __forceinline__ int64_t src_row(int64_t p, int64_t Sb, int64_t N, int layout,
                                           int inverse) {
    return inverse ? row_of_token(p, Sb, N, layout) : token_of_row(p, Sb, N, layout);
}

template <typename V>
__global__ void __launch_bounds__(kBlock) stripe_kernel(const V* __restrict__ src, V* __restrict__ dst,
                                                        int64_t BH, int64_t S, int64_t N,
                                                        int64_t row_vecs, int layout, int inverse) {
    const int lane = threadIdx.x & 31;
    const int64_t Sb = S / N;
    const int64_t total = BH * S;
    const int64_t warps = (int64_t)gridDim.x * (kBlock / 32);
    for (int64_t wr = (int64_t)blockIdx.x * (kBlock / 32) + threadIdx.x / 32; wr < total;
         wr += warps) {
        const int64_t bh = wr / S, p = wr % S;  // p: destination row within the slice
        const int64_t sp = src_row(p, Sb, N, layout, inverse);
        const V* s = src + (bh * S + sp) * row_vecs;
        V* d = dst + (bh * S + p) * row_vecs;
        for (int64_t e = lane; e < row_vecs; e += 32) d[e] = s[e];
    }
}

// Row-group variants: a row of VPR 16-byte vectors (VPR a power of two <= 32)
// is handled by VPR consecutive lanes, so a warp covers 32/VPR rows at once
// and every lane moves 16 bytes; UNROLL batches are loaded before any store
// to keep enough bytes in flight for HBM.
template <typename T, int VPR, int UNROLL>
__global__ void __launch_bounds__(kBlock) merge_rows_kernel(T* __restrict__ oa, float* __restrict__ la,
                                                           const T* __restrict__ ob,
                                                           const float* __restrict__ lb,
                                                           int64_t rows) {
    constexpr int RPW = 32 / VPR;  // rows per warp per batch
    const int lane = threadIdx.x & 31, sub = lane / VPR, v = lane % VPR;
    const int64_t warp_id = ((int64_t)blockIdx.x * kBlock + threadIdx.x) / 32;
    const int64_t n_warps = (int64_t)gridDim.x * (kBlock / 32);
    uint4* va = reinterpret_cast<uint4*>(oa);
    const uint4* vb = reinterpret_cast<const uint4*>(ob);
    for (int64_t r0 = warp_id * RPW * UNROLL; r0 < rows; r0 += n_warps * RPW * UNROLL) {
        uint4 xa[UNROLL], xb[UNROLL];
        float ca[UNROLL], cb[UNROLL], ls[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t row = r0 + u * RPW + sub;
            if (row < rows) {
                xa[u] = va[row * VPR + v];
                xb[u] = __ldg(vb + row * VPR + v);
                const float a = la[row], b = __ldg(lb + row);
                const float mx = fmaxf(a, b);
                ca[u] = cb[u] = 0.f;
                ls[u] = -INFINITY;
                if (mx != -INFINITY) {
                    const float wa = expf(a - mx), wb = expf(b - mx), tot = wa + wb;
                    ls[u] = mx + logf(tot);
                    ca[u] = wa / tot;
                    cb[u] = wb / tot;
                }
            }
        }
        __syncwarp();  // every lane has read la[] before lane 0 of a row rewrites it
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t row = r0 + u * RPW + sub;
            if (row < rows) {
                Vec<T>::fma2(xa[u], xb[u], ca[u], cb[u]);
                va[row * VPR + v] = xa[u];
                if (v == 0) la[row] = ls[u];  // every lane of this row read la[row] above
            }
        }
    }
}

template <int VPR, int UNROLL>
__global__ void __launch_bounds__(kBlock) stripe_rows_kernel(const uint4* __restrict__ src,
                                                            uint4* __restrict__ dst, int64_t BH,
                                                            int64_t S, int64_t N, int layout,
                                                            int inverse) {
    constexpr int RPW = 32 / VPR;
    const int lane = threadIdx.x & 31, sub = lane / VPR, v = lane % VPR;
    const int64_t Sb = S / N, total = BH * S;
    const int64_t warp_id = ((int64_t)blockIdx.x * kBlock + threadIdx.x) / 32;
    const int64_t n_warps = (int64_t)gridDim.x * (kBlock / 32);
    for (int64_t r0 = warp_id * RPW * UNROLL; r0 < total; r0 += n_warps * RPW * UNROLL) {
        uint4 x[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t wr = r0 + u * RPW + sub;
            if (wr < total) {
                const int64_t bh = wr / S, p = wr % S;
                const int64_t sp = src_row(p, Sb, N, layout, inverse);
                x[u] = __ldg(src + (bh * S + sp) * VPR + v);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t wr = r0 + u * RPW + sub;
            if (wr < total) dst[wr * VPR + v] = x[u];
        }
    }
}

// Ulysses head/sequence exchange between N device-contiguous buffers:
// forward, sequence-sharded [N][B][H][Sb] -> head-sharded [N][B][H/N][S]:
//   dst[d][b][hl][t] = src[t / Sb][b][d*H/N + hl][t % Sb]; inverse maps back.
// The exchange moves whole chunks of Sb consecutive rows: destination chunk c
// (grid y) is decoded once per thread, then its Sb*row_bytes bytes are copied
// as 16-byte vectors (or 4-byte words when rows are not 16-byte multiples).
template <typename V>
__global__ void __launch_bounds__(kBlock) ulysses_chunks_kernel(const V* __restrict__ src,
                                                               V* __restrict__ dst, int64_t B,
                                                               int64_t H, int64_t S, int64_t N,
                                                               int64_t chunk_elems, int inverse) {
    const int64_t c = blockIdx.y;  // destination chunk
    const int64_t Hl = H / N;
    int64_t src_chunk_row;         // first source row of the chunk
    if (!inverse) {                // c = ((d*B + b)*Hl + hl)*N + i
        const int64_t i = c % N, hl = (c / N) % Hl, b = (c / (N * Hl)) % B, d = c / (N * Hl * B);
        src_chunk_row = ((i * B + b) * H + d * Hl + hl) * (S / N);
    } else {                       // c = (i*B + b)*H + h
        const int64_t h = c % H, b = (c / H) % B, i = c / (H * B);
        src_chunk_row = ((h / Hl * B + b) * Hl + h % Hl) * S + i * (S / N);
    }
    const int64_t row_elems = chunk_elems / (S / N);
    const V* s = src + src_chunk_row * row_elems;
    V* d = dst + c * chunk_elems;
    constexpr int U = 4;
    for (int64_t e = ((int64_t)blockIdx.x * kBlock + threadIdx.x) * U; e < chunk_elems;
         e += (int64_t)gridDim.x * kBlock * U) {
        V x[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (e + u < chunk_elems) x[u] = __ldg(s + e + u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (e + u < chunk_elems) d[e + u] = x[u];
    }
}

static unsigned grid_for(int64_t rows) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t need = (rows + (kBlock / 32) - 1) / (kBlock / 32);
    const int64_t cap = (int64_t)sms * 16;
    return (unsigned)(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace aux

int launch_ulysses(const void* src, void* dst, int64_t B, int64_t H, int64_t S, int N,
                   int64_t row_bytes, int inverse, cudaStream_t stream) {
    const int64_t chunks = B * H * N;
    if (chunks == 0 || S == 0) return RA_OK;
    if (chunks > 65535) {  // one grid row per chunk
        return RA_ERR_UNSUPPORTED;
    }
    const int64_t chunk_bytes = (S / N) * row_bytes;
    const bool vec = (row_bytes % 16 == 0);
    const int64_t chunk_elems = chunk_bytes / (vec ? 16 : 4);
    int64_t gx = (chunk_elems + aux::kBlock * 4 - 1) / (aux::kBlock * 4);
    if (gx > 64) gx = 64;
    if (gx < 1) gx = 1;
    dim3 grid((unsigned)gx, (unsigned)chunks);
    if (vec)
        aux::ulysses_chunks_kernel<uint4><<<grid, aux::kBlock, 0, stream>>>(
            static_cast<const uint4*>(src), static_cast<uint4*>(dst), B, H, S, N, chunk_elems,
            inverse);
    else
        aux::ulysses_chunks_kernel<uint32_t><<<grid, aux::kBlock, 0, stream>>>(
            static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), B, H, S, N,
            chunk_elems, inverse);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

int launch_merge(void* out_a, float* lse_a, const void* out_b, const float* lse_b, int64_t rows,
                 int D, int dtype, cudaStream_t stream) {
    if (rows == 0) return RA_OK;
    const unsigned grid = aux::grid_for(rows);
    if (dtype == RA_BF16 && (D == 64 || D == 128 || D == 256)) {
        auto* a = static_cast<__nv_bfloat16*>(out_a);
        auto* b = static_cast<const __nv_bfloat16*>(out_b);
        const unsigned g = aux::grid_for(rows / 8 + 1);
        if (D == 64) aux::merge_rows_kernel<__nv_bfloat16, 8, 4><<<g, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows);
        else if (D == 128) aux::merge_rows_kernel<__nv_bfloat16, 16, 4><<<g, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows);
        else aux::merge_rows_kernel<__nv_bfloat16, 32, 4><<<g, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows);
    } else if (dtype == RA_BF16) {
        auto* a = static_cast<__nv_bfloat16*>(out_a);
        auto* b = static_cast<const __nv_bfloat16*>(out_b);
        if (D % 8 == 0)
            aux::merge_kernel<__nv_bfloat16, true><<<grid, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows, D);
        else
            aux::merge_kernel<__nv_bfloat16, false><<<grid, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows, D);
    } else {
        auto* a = static_cast<float*>(out_a);
        auto* b = static_cast<const float*>(out_b);
        if (D % 4 == 0)
            aux::merge_kernel<float, true><<<grid, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows, D);
        else
            aux::merge_kernel<float, false><<<grid, aux::kBlock, 0, stream>>>(a, lse_a, b, lse_b, rows, D);
    }
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

int launch_stripe(const void* src, void* dst, int64_t BH, int64_t S, int N, int64_t row_bytes,
                  int layout, int inverse, cudaStream_t stream) {
    const int64_t rows = BH * S;
    if (rows == 0) return RA_OK;
    const unsigned grid = aux::grid_for(rows);
    const int64_t vpr = row_bytes / 16;
    if (row_bytes % 16 == 0 && (vpr == 2 || vpr == 4 || vpr == 8 || vpr == 16 || vpr == 32)) {
        const unsigned g = aux::grid_for(rows / 8 + 1);
        auto* sp = static_cast<const uint4*>(src);
        auto* dp = static_cast<uint4*>(dst);
        switch (vpr) {
            case 2: aux::stripe_rows_kernel<2, 4><<<g, aux::kBlock, 0, stream>>>(sp, dp, BH, S, N, layout, inverse); break;
            case 4: aux::stripe_rows_kernel<4, 4><<<g, aux::kBlock, 0, stream>>>(sp, dp, BH, S, N, layout, inverse); break;
            case 8: aux::stripe_rows_kernel<8, 4><<<g, aux::kBlock, 0, stream>>>(sp, dp, BH, S, N, layout, inverse); break;
            case 16: aux::stripe_rows_kernel<16, 4><<<g, aux::kBlock, 0, stream>>>(sp, dp, BH, S, N, layout, inverse); break;
            default: aux::stripe_rows_kernel<32, 4><<<g, aux::kBlock, 0, stream>>>(sp, dp, BH, S, N, layout, inverse); break;
        }
    } else if (row_bytes % 16 == 0)
        aux::stripe_kernel<uint4><<<grid, aux::kBlock, 0, stream>>>(
            static_cast<const uint4*>(src), static_cast<uint4*>(dst), BH, S, N, row_bytes / 16, layout, inverse);
    else
        aux::stripe_kernel<uint32_t><<<grid, aux::kBlock, 0, stream>>>(
            static_cast<const uint32_t*>(src), static_cast<uint32_t*>(dst), BH, S, N, row_bytes / 4, layout, inverse);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

}  // namespace ra
