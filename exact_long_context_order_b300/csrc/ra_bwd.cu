// Ring-attention backward: the per-row terms delta and the fp32 SIMT backward
// (f32 or bf16 tensors, fp32 FFMA, no TF32, D <= 128, any shard size).
//
// The gradients are the chain rule of O = softmax(scale Q K^T) V (the pages
// use the method for training -- the Italian aiunderstanding.org page,
// "Implementazione nel mondo reale", and the glossary page's training
// throughput remark -- without writing the backward out).  With
// P_tu = exp(scale q_t.k_u - lse_t) over the visible pairs and
// delta_t = dO_t . O_t:
//   dS_tu = P_tu (dO_t . v_u - delta_t)
//   dq_t  = scale sum_u dS_tu k_u
//   dk_u  = scale sum_t dS_tu q_t       dv_u = sum_t P_tu dO_t
// The dq kernel gives each thread one query row of shard i and walks the
// key/value shards in the forward's ring order j = (i - s) mod N.  The dk/dv
// kernel gives each thread one key row of shard j; its accumulators travel
// with the block like the block itself, visiting query shards
// i = (j + s) mod N, s = 0..N-1, and within each the query heads of its GQA
// group (the tensor-core kernel enters the same cyclic order at device 0).  Visibility comes from token positions, as in the SIMT forward.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ra.h"

namespace ra {
namespace bwd {

constexpr int kRows = 128;

struct Params {
    int B, Hq, Hkv, g, N, D, causal, layout;
    int64_t S, Sb;
    float scale;
};

// token position of local row r of shard i (0 contiguous, 1 striped, 2 zigzag)
__device__ __forceinline__ int64_t token_pos(const Params& p, int64_t i, int64_t r) {
    if (p.layout == 1) return r * p.N + i;
    if (p.layout == 2) {
        const int64_t h = p.Sb / 2;
        return r < h ? i * h + r : (2 * (int64_t)p.N - 1 - i) * h + (r - h);
    }
    return i * p.Sb + r;
}

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// delta[row] = sum_d dout[row, d] * out[row, d]; one warp per row.
template <typename T>
__global__ void __launch_bounds__(256) delta_kernel(const T* __restrict__ out,
                                                    const T* __restrict__ dout,
                                                    float* __restrict__ delta, int64_t rows,
                                                    int D) {
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const T* o = out + row * D;
    const T* g = dout + row * D;
    float acc = 0.f;
    for (int d = lane; d < D; d += 32) acc = fmaf(load_f(o + d), load_f(g + d), acc);
#pragma unroll
    for (int w = 16; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (lane == 0) delta[row] = acc;
}

// bf16 D = 128: sixteen lanes per row, eight elements (16 bytes) per lane.
__global__ void __launch_bounds__(256) delta_bf16_d128_kernel(const uint4* __restrict__ out,
                                                              const uint4* __restrict__ dout,
                                                              float* __restrict__ delta,
                                                              int64_t rows) {
    const int64_t row = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);
    const int part = threadIdx.x & 15;
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = out[row * 16 + part];
        const uint4 b = dout[row * 16 + part];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
            const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[e]));
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
#pragma unroll
    for (int w = 8; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (row < rows && part == 0) delta[row] = acc;
}

template <typename T, int DMAX, int KC>
__global__ void __launch_bounds__(kRows) dq_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                   const T* __restrict__ v,
                                                   const T* __restrict__ dout,
                                                   const float* __restrict__ lse,
                                                   const float* __restrict__ delta,
                                                   T* __restrict__ dq, const Params p) {
    __shared__ float ks[KC][DMAX];
    __shared__ float vs[KC][DMAX];
    const int i = blockIdx.y;
    const int bh = blockIdx.z;
    const int b = bh / p.Hq, h = bh % p.Hq;
    const int kvh = h / p.g;
    const int64_t r0 = (int64_t)blockIdx.x * kRows;
    const int64_t r = r0 + threadIdx.x;
    const int64_t r_last = (r0 + kRows - 1 < p.Sb) ? r0 + kRows - 1 : p.Sb - 1;
    const int64_t N = p.N;
    const int64_t qpos = token_pos(p, i, r);
    const int64_t qpos_last = token_pos(p, i, r_last);
    const int D = p.D;
    const int64_t row = (int64_t)bh * p.S + i * p.Sb + (r < p.Sb ? r : 0);
    const float L = lse[row];
    const bool active = r < p.Sb && L > -INFINITY;
    const float dl = delta[row];

    float qr[DMAX], gr[DMAX], acc[DMAX];
#pragma unroll
    for (int d = 0; d < DMAX; ++d) {
        qr[d] = (d < D) ? load_f(q + row * D + d) * p.scale : 0.f;
        gr[d] = (d < D) ? load_f(dout + row * D + d) : 0.f;
        acc[d] = 0.f;
    }
    const T* kbase = k + ((int64_t)b * p.Hkv + kvh) * p.S * D;
    const T* vbase = v + ((int64_t)b * p.Hkv + kvh) * p.S * D;

    for (int s = 0; s < p.N; ++s) {
        const int j = (int)((i - s + N) % N);
        for (int64_t c0 = 0; c0 < p.Sb; c0 += KC) {
            if (p.causal && token_pos(p, j, c0) > qpos_last) break;
            const int nk = (int)((p.Sb - c0 < KC) ? p.Sb - c0 : KC);
            __syncthreads();
            for (int e = threadIdx.x; e < KC * DMAX; e += kRows) {
                const int kr = e / DMAX, d = e % DMAX;
                float kv = 0.f, vv = 0.f;
                if (kr < nk && d < D) {
                    const int64_t off = (j * p.Sb + c0 + kr) * D + d;
                    kv = load_f(kbase + off);
                    vv = load_f(vbase + off);
                }
                ks[kr][d] = kv;
                vs[kr][d] = vv;
            }
            __syncthreads();
            if (!active) continue;
            for (int kr = 0; kr < nk; ++kr) {
                if (p.causal && token_pos(p, j, c0 + kr) > qpos) continue;
                float sc = 0.f, dp = 0.f;
#pragma unroll
                for (int d = 0; d < DMAX; ++d) {
                    sc = fmaf(qr[d], ks[kr][d], sc);
                    dp = fmaf(gr[d], vs[kr][d], dp);
                }
                const float ds = expf(sc - L) * (dp - dl);
#pragma unroll
                for (int d = 0; d < DMAX; ++d) acc[d] = fmaf(ds, ks[kr][d], acc[d]);
            }
        }
    }
    if (r >= p.Sb) return;
#pragma unroll
    for (int d = 0; d < DMAX; ++d)
        if (d < D) store_f(dq + row * D + d, active ? acc[d] * p.scale : 0.f);
}

template <typename T, int DMAX, int QC>
__global__ void __launch_bounds__(kRows) dkdv_kernel(const T* __restrict__ q,
                                                     const T* __restrict__ k,
                                                     const T* __restrict__ v,
                                                     const T* __restrict__ dout,
                                                     const float* __restrict__ lse,
                                                     const float* __restrict__ delta,
                                                     T* __restrict__ dk, T* __restrict__ dv,
                                                     const Params p) {
    __shared__ float qs[QC][DMAX];
    __shared__ float gs[QC][DMAX];
    __shared__ float ls[QC], dls[QC];
    const int j = blockIdx.y;  // key/value shard
    const int bk = blockIdx.z;  // b * Hkv + kv head
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int64_t u0 = (int64_t)blockIdx.x * kRows;
    const int64_t u = u0 + threadIdx.x;
    const bool active = u < p.Sb;
    const int64_t N = p.N;
    const int64_t kpos = token_pos(p, j, active ? u : u0);
    const int64_t kpos_first = token_pos(p, j, u0);  // smallest key position of the block
    const int D = p.D;
    const int64_t krow = (int64_t)bk * p.S + j * p.Sb + (active ? u : 0);

    float kr[DMAX], vr[DMAX], dka[DMAX], dva[DMAX];
#pragma unroll
    for (int d = 0; d < DMAX; ++d) {
        kr[d] = (d < D) ? load_f(k + krow * D + d) : 0.f;
        vr[d] = (d < D) ? load_f(v + krow * D + d) : 0.f;
        dka[d] = 0.f;
        dva[d] = 0.f;
    }

    for (int s = 0; s < p.N; ++s) {
        const int i = (int)((j + s) % N);  // query shard the block visits at step s
        for (int gi = 0; gi < p.g; ++gi) {
            const int64_t bh = (int64_t)b * p.Hq + (int64_t)kvh * p.g + gi;
            const int64_t qbase = bh * p.S + i * p.Sb;
            for (int64_t c0 = 0; c0 < p.Sb; c0 += QC) {
                const int nq = (int)((p.Sb - c0 < QC) ? p.Sb - c0 : QC);
                // query positions ascend within a shard: a chunk whose last
                // row precedes every key of the block has no visible pair
                if (p.causal && token_pos(p, i, c0 + nq - 1) < kpos_first) continue;
                __syncthreads();
                for (int e = threadIdx.x; e < QC * DMAX; e += kRows) {
                    const int qr = e / DMAX, d = e % DMAX;
                    float qv = 0.f, gv = 0.f;
                    if (qr < nq && d < D) {
                        const int64_t off = (qbase + c0 + qr) * D + d;
                        qv = load_f(q + off);
                        gv = load_f(dout + off);
                    }
                    qs[qr][d] = qv;
                    gs[qr][d] = gv;
                }
                if (threadIdx.x < QC) {
                    const bool ok = threadIdx.x < nq;
                    ls[threadIdx.x] = ok ? lse[qbase + c0 + threadIdx.x] : -INFINITY;
                    dls[threadIdx.x] = ok ? delta[qbase + c0 + threadIdx.x] : 0.f;
                }
                __syncthreads();
                if (!active) continue;
                for (int qr = 0; qr < nq; ++qr) {
                    if (p.causal && token_pos(p, i, c0 + qr) < kpos) continue;
                    const float L = ls[qr];
                    if (!(L > -INFINITY)) continue;
                    float sc = 0.f, dp = 0.f;
#pragma unroll
                    for (int d = 0; d < DMAX; ++d) {
                        sc = fmaf(qs[qr][d], kr[d], sc);
                        dp = fmaf(gs[qr][d], vr[d], dp);
                    }
                    const float pe = expf(sc * p.scale - L);
                    const float ds = pe * (dp - dls[qr]);
#pragma unroll
                    for (int d = 0; d < DMAX; ++d) {
                        dva[d] = fmaf(pe, gs[qr][d], dva[d]);
                        dka[d] = fmaf(ds, qs[qr][d], dka[d]);
                    }
                }
            }
        }
    }
    if (!active) return;
#pragma unroll
    for (int d = 0; d < DMAX; ++d)
        if (d < D) {
            store_f(dk + krow * D + d, dka[d] * p.scale);
            store_f(dv + krow * D + d, dva[d]);
        }
}

Params make_params(const BwdProblem& pr) {
    Params P;
    P.B = pr.B; P.Hq = pr.Hq; P.Hkv = pr.Hkv; P.g = pr.Hq / pr.Hkv; P.N = pr.N; P.D = pr.D;
    P.causal = pr.causal; P.layout = pr.striped;
    P.S = pr.S; P.Sb = pr.S / pr.N;
    P.scale = pr.scale;
    return P;
}

template <typename T, int DMAX>
int launch_simt_t(const BwdProblem& pr, cudaStream_t stream) {
    const Params P = make_params(pr);
    constexpr int KC = (DMAX <= 64) ? 32 : 16;
    const unsigned bx = (unsigned)((P.Sb + kRows - 1) / kRows);
    dq_kernel<T, DMAX, KC><<<dim3(bx, pr.N, pr.B * pr.Hq), kRows, 0, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<const T*>(pr.dout), pr.lse, pr.delta, static_cast<T*>(pr.dq), P);
    if (cudaGetLastError() != cudaSuccess) return RA_ERR_CUDA;
    dkdv_kernel<T, DMAX, KC><<<dim3(bx, pr.N, pr.B * pr.Hkv), kRows, 0, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<const T*>(pr.dout), pr.lse, pr.delta, static_cast<T*>(pr.dk),
        static_cast<T*>(pr.dv), P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

template <typename T, int DMAX>
int launch_dkdv_t(const BwdProblem& pr, cudaStream_t stream) {
    const Params P = make_params(pr);
    constexpr int KC = (DMAX <= 64) ? 32 : 16;
    const unsigned bx = (unsigned)((P.Sb + kRows - 1) / kRows);
    dkdv_kernel<T, DMAX, KC><<<dim3(bx, pr.N, pr.B * pr.Hkv), kRows, 0, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<const T*>(pr.dout), pr.lse, pr.delta, static_cast<T*>(pr.dk),
        static_cast<T*>(pr.dv), P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

template <typename T>
int launch_simt_d(const BwdProblem& pr, cudaStream_t stream) {
    if (pr.D <= 32) return launch_simt_t<T, 32>(pr, stream);
    if (pr.D <= 64) return launch_simt_t<T, 64>(pr, stream);
    return launch_simt_t<T, 128>(pr, stream);
}

}  // namespace bwd

bool bwd_delta_supported(const BwdProblem& p) {
    return ((int64_t)p.B * p.Hq * p.S + 7) / 8 <= 0x7fffffff;
}

bool simt_bwd_supported(const BwdProblem& p) {
    // grids (row blocks, N, B*Hq) and (row blocks, N, B*Hkv)
    return p.D <= 128 && (int64_t)p.B * p.Hq <= 65535 && (int64_t)p.B * p.Hkv <= 65535 &&
           p.N <= 65535 && (p.S / p.N + 127) / 128 <= 0x7fffffff;
}

int launch_bwd_delta(const BwdProblem& p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.Hq * p.S;
    if (rows == 0) return RA_OK;
    if (p.dtype == RA_BF16 && p.D == 128) {
        const int64_t blocks = (rows + 15) / 16;
        if (blocks > 0x7fffffff) return RA_ERR_UNSUPPORTED;
        bwd::delta_bf16_d128_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const uint4*>(p.out), static_cast<const uint4*>(p.dout), p.delta, rows);
    } else {
        const int64_t blocks = (rows + 7) / 8;
        if (blocks > 0x7fffffff) return RA_ERR_UNSUPPORTED;
        if (p.dtype == RA_F32)
            bwd::delta_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(
                static_cast<const float*>(p.out), static_cast<const float*>(p.dout), p.delta,
                rows, p.D);
        else
            bwd::delta_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16*>(p.out),
                static_cast<const __nv_bfloat16*>(p.dout), p.delta, rows, p.D);
    }
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

int launch_bwd_simt(const BwdProblem& p, cudaStream_t stream) {
    if (p.D > 128) return RA_ERR_UNSUPPORTED;
    if ((int64_t)p.B * p.Hq > 65535 || p.N > 65535 || (p.S / p.N + 127) / 128 > 0x7fffffff)
        return RA_ERR_UNSUPPORTED;
    return p.dtype == RA_F32 ? bwd::launch_simt_d<float>(p, stream)
                             : bwd::launch_simt_d<__nv_bfloat16>(p, stream);
}

int launch_bwd_dkdv_simt(const BwdProblem& p, cudaStream_t stream) {
    if (p.D > 128 || (int64_t)p.B * p.Hkv > 65535 || p.N > 65535) return RA_ERR_UNSUPPORTED;
    if (p.dtype == RA_F32) return bwd::launch_dkdv_t<float, 128>(p, stream);
    return bwd::launch_dkdv_t<__nv_bfloat16, 128>(p, stream);
}

}  // namespace ra
