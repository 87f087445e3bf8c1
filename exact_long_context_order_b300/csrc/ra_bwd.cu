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

// ---------------------------------------------------------------- tiled kernels (D % 4 == 0, D <= 128)
// Register-blocked versions of the two kernels above, for D % 4 == 0 and
// D <= 128 (DMAX = 32, 64 or 128, D padded by zeros); the fold orders are
// the same.  A block holds 64 rows of its own side (query rows for dq, key
// rows for dk/dv) transposed in shared memory and streams the other side in
// chunks of 32 rows, stored row-major in rows padded to DMAX + 4 floats.
// Thread (rg, kg) = (tid / 8, tid % 8) computes the 4 x 4 products of its
// rows 4rg..4rg+3 with chunk rows kg, kg+8, kg+16, kg+24 (the padding puts
// the eight kg lanes on different bank groups), and accumulates its rows'
// gradients on dims {32t + 4kg + e}.
constexpr int kTR = 64;       // rows of the block's own side
constexpr int kTK = 32;       // rows per chunk of the other side
constexpr int kTThreads = 128;

__device__ __forceinline__ void load4_f(const float* p, float* x) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
}
__device__ __forceinline__ void load4_f(const __nv_bfloat16* p, float* x) {
    const uint2 t = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(t.x << 16); x[1] = __uint_as_float(t.x & 0xffff0000u);
    x[2] = __uint_as_float(t.y << 16); x[3] = __uint_as_float(t.y & 0xffff0000u);
}
__device__ __forceinline__ void store4_f(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store4_f(__nv_bfloat16* p, const float* x) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 t;
    t.x = *reinterpret_cast<const uint32_t*>(&a);
    t.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = t;
}

// rows [r0, r0 + 64) of a [rows, D] matrix, transposed into dst[DMAX][64]
// and multiplied by mul; rows at or past `valid` and dims past D are zero
template <typename T, int DMAX>
__device__ __forceinline__ void stage_transposed(float (*dst)[kTR], const T* src, int64_t r0,
                                                 int64_t valid, int D, float mul) {
    for (int e = threadIdx.x; e < kTR * (DMAX / 4); e += kTThreads) {
        const int r = e % kTR, d4 = e / kTR;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (r0 + r < valid && 4 * d4 < D) load4_f(src + (r0 + r) * D + 4 * d4, x);
#pragma unroll
        for (int a = 0; a < 4; ++a) dst[4 * d4 + a][r] = x[a] * mul;
    }
}
// rows [c0, c0 + n) of a [rows, D] matrix into dst[32][DMAX + 4]; the rest zero
template <typename T, int DMAX>
__device__ __forceinline__ void stage_rows(float (*dst)[DMAX + 4], const T* src, int64_t c0, int n,
                                           int D) {
    for (int e = threadIdx.x; e < kTK * (DMAX / 4); e += kTThreads) {
        const int d4 = e % (DMAX / 4), r = e / (DMAX / 4);
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < n && 4 * d4 < D) load4_f(src + (c0 + r) * D + 4 * d4, x);
        store4_f(&dst[r][4 * d4], x);
    }
}
// acc[a][c] += sum_d A[d][4rg + a] * Brows[kg + 8c][d]
template <int DMAX>
__device__ __forceinline__ void block_products(float (&acc)[4][4], const float (*A)[kTR],
                                               const float (*Brows)[DMAX + 4], int rg, int kg) {
#pragma unroll 2
    for (int d4 = 0; d4 < DMAX / 4; ++d4) {
        float av[4][4], bv[4][4];  // [dim][row], [chunk row][dim]
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 t = *reinterpret_cast<const float4*>(&A[4 * d4 + e][4 * rg]);
            av[e][0] = t.x; av[e][1] = t.y; av[e][2] = t.z; av[e][3] = t.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float4 t = *reinterpret_cast<const float4*>(&Brows[kg + 8 * c][4 * d4]);
            bv[c][0] = t.x; bv[c][1] = t.y; bv[c][2] = t.z; bv[c][3] = t.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(av[e][a], bv[c][e], acc[a][c]);
    }
}

template <int DMAX>
struct DqSmem {
    float qt[DMAX][kTR];        // scale * q, transposed
    float gt[DMAX][kTR];        // dout, transposed
    float ks[kTK][DMAX + 4];    // k rows of the chunk
    float vs[kTK][DMAX + 4];    // v rows of the chunk
    float ps[kTR][kTK + 1];     // dS of the chunk
};

template <typename T, int DMAX>
__global__ void __launch_bounds__(kTThreads)
    dq_tiled_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    const T* __restrict__ dout, const float* __restrict__ lse,
                    const float* __restrict__ delta, T* __restrict__ dq, const Params p) {
    constexpr int DPT = DMAX / 8;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    DqSmem<DMAX>& sm = *reinterpret_cast<DqSmem<DMAX>*>(smem_raw);
    const int tid = threadIdx.x, rg = tid >> 3, kg = tid & 7;
    const int i = blockIdx.y;   // query shard
    const int bh = blockIdx.z;  // b * Hq + h
    const int b = bh / p.Hq, h = bh % p.Hq, kvh = h / p.g;
    const int64_t r0 = (int64_t)blockIdx.x * kTR;
    const int64_t N = p.N, Sb = p.Sb;
    const int D = p.D;
    const int64_t r_last = (r0 + kTR - 1 < Sb) ? r0 + kTR - 1 : Sb - 1;
    const int64_t qpos_last = token_pos(p, i, r_last);
    const int64_t rowbase = (int64_t)bh * p.S + i * Sb;
    int64_t qpos[4];
    float L[4], dl[4];
    bool rok[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t r = r0 + 4 * rg + a;
        qpos[a] = token_pos(p, i, r);
        L[a] = (r < Sb) ? lse[rowbase + r] : -INFINITY;
        dl[a] = (r < Sb) ? delta[rowbase + r] : 0.f;
        rok[a] = r < Sb && L[a] > -INFINITY;
    }
    stage_transposed<T, DMAX>(sm.qt, q + rowbase * D, r0, Sb, D, p.scale);
    stage_transposed<T, DMAX>(sm.gt, dout + rowbase * D, r0, Sb, D, 1.f);
    float acc[4][DPT];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int d = 0; d < DPT; ++d) acc[a][d] = 0.f;
    const T* kbase = k + ((int64_t)b * p.Hkv + kvh) * p.S * D;
    const T* vbase = v + ((int64_t)b * p.Hkv + kvh) * p.S * D;

    for (int s = 0; s < p.N; ++s) {
        const int j = (int)((i - s + N) % N);
        for (int64_t c0 = 0; c0 < Sb; c0 += kTK) {
            if (p.causal && token_pos(p, j, c0) > qpos_last) break;  // keys ascend in a shard
            const int nk = (int)((Sb - c0 < kTK) ? Sb - c0 : kTK);
            __syncthreads();  // the previous chunk's reads are done
            stage_rows<T, DMAX>(sm.ks, kbase + j * Sb * D, c0, nk, D);
            stage_rows<T, DMAX>(sm.vs, vbase + j * Sb * D, c0, nk, D);
            __syncthreads();
            float sc[4][4], dp[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[a][c] = dp[a][c] = 0.f;
            block_products<DMAX>(sc, sm.qt, sm.ks, rg, kg);
            block_products<DMAX>(dp, sm.gt, sm.vs, rg, kg);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = kg + 8 * c;
                const int64_t kpos = token_pos(p, j, c0 + key);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const bool vis = rok[a] && key < nk && !(p.causal && kpos > qpos[a]);
                    sm.ps[4 * rg + a][key] = vis ? expf(sc[a][c] - L[a]) * (dp[a][c] - dl[a]) : 0.f;
                }
            }
            __syncthreads();
            // dq += dS k on dims {32t + 4kg + e}
#pragma unroll 4
            for (int key = 0; key < kTK; ++key) {
                float dsr[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) dsr[a] = sm.ps[4 * rg + a][key];
#pragma unroll
                for (int t = 0; t < DPT / 4; ++t) {
                    const float4 kk = *reinterpret_cast<const float4*>(&sm.ks[key][32 * t + 4 * kg]);
                    const float kx[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc[a][4 * t + e] = fmaf(dsr[a], kx[e], acc[a][4 * t + e]);
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t r = r0 + 4 * rg + a;
        if (r >= Sb) continue;
#pragma unroll
        for (int t = 0; t < DPT / 4; ++t) {
            const int d0 = 32 * t + 4 * kg;
            if (d0 >= D) continue;
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = rok[a] ? acc[a][4 * t + e] * p.scale : 0.f;
            store4_f(dq + (rowbase + r) * D + d0, x);
        }
    }
}

template <int DMAX>
struct DkvSmem {
    float kt[DMAX][kTR];        // scale * k, transposed (the block's keys)
    float vt[DMAX][kTR];        // v, transposed
    float qs[kTK][DMAX + 4];    // q rows of the chunk
    float gs[kTK][DMAX + 4];    // dout rows of the chunk
    float pt[kTR][kTK + 1];     // P^T of the chunk
    float dst[kTR][kTK + 1];    // dS^T of the chunk
    float ls[kTK], dls[kTK];    // lse and delta of the chunk's query rows
};

template <typename T, int DMAX>
__global__ void __launch_bounds__(kTThreads)
    dkdv_tiled_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const T* __restrict__ dout, const float* __restrict__ lse,
                      const float* __restrict__ delta, T* __restrict__ dk, T* __restrict__ dv,
                      const Params p) {
    constexpr int DPT = DMAX / 8;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    DkvSmem<DMAX>& sm = *reinterpret_cast<DkvSmem<DMAX>*>(smem_raw);
    const int tid = threadIdx.x, rg = tid >> 3, kg = tid & 7;
    const int j = blockIdx.y;   // key/value shard
    const int bk = blockIdx.z;  // b * Hkv + kv head
    const int b = bk / p.Hkv, kvh = bk % p.Hkv;
    const int64_t u0 = (int64_t)blockIdx.x * kTR;
    const int64_t N = p.N, Sb = p.Sb;
    const int D = p.D;
    const int64_t kpos_first = token_pos(p, j, u0);  // smallest key position of the block
    const int64_t keybase = (int64_t)bk * p.S + j * Sb;
    int64_t kpos[4];
    bool kok[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t u = u0 + 4 * rg + a;
        kpos[a] = token_pos(p, j, u);
        kok[a] = u < Sb;
    }
    stage_transposed<T, DMAX>(sm.kt, k + keybase * D, u0, Sb, D, p.scale);
    stage_transposed<T, DMAX>(sm.vt, v + keybase * D, u0, Sb, D, 1.f);
    float dka[4][DPT], dva[4][DPT];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int d = 0; d < DPT; ++d) dka[a][d] = dva[a][d] = 0.f;

    for (int s = 0; s < p.N; ++s) {
        const int i = (int)((j + s) % N);  // query shard the block visits at step s
        for (int gi = 0; gi < p.g; ++gi) {
            const int64_t bh = (int64_t)b * p.Hq + (int64_t)kvh * p.g + gi;
            const int64_t qbase = bh * p.S + i * Sb;
            for (int64_t c0 = 0; c0 < Sb; c0 += kTK) {
                const int nq = (int)((Sb - c0 < kTK) ? Sb - c0 : kTK);
                // query positions ascend within a shard: a chunk whose last
                // row precedes every key of the block has no visible pair
                if (p.causal && token_pos(p, i, c0 + nq - 1) < kpos_first) continue;
                __syncthreads();  // the previous chunk's reads are done
                stage_rows<T, DMAX>(sm.qs, q + qbase * D, c0, nq, D);
                stage_rows<T, DMAX>(sm.gs, dout + qbase * D, c0, nq, D);
                if (tid < kTK) {
                    sm.ls[tid] = (tid < nq) ? lse[qbase + c0 + tid] : -INFINITY;
                    sm.dls[tid] = (tid < nq) ? delta[qbase + c0 + tid] : 0.f;
                }
                __syncthreads();
                float sc[4][4], dp[4][4];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sc[a][c] = dp[a][c] = 0.f;
                block_products<DMAX>(sc, sm.kt, sm.qs, rg, kg);
                block_products<DMAX>(dp, sm.vt, sm.gs, rg, kg);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int qq = kg + 8 * c;
                    const int64_t qpos = token_pos(p, i, c0 + qq);
                    const float Lq = sm.ls[qq], dq_ = sm.dls[qq];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const bool vis = kok[a] && qq < nq && Lq > -INFINITY &&
                                         !(p.causal && qpos < kpos[a]);
                        const float pe = vis ? expf(sc[a][c] - Lq) : 0.f;
                        sm.pt[4 * rg + a][qq] = pe;
                        sm.dst[4 * rg + a][qq] = pe * (dp[a][c] - dq_);
                    }
                }
                __syncthreads();
                // dv += P^T dout, dk += dS^T q on dims {32t + 4kg + e}
#pragma unroll 2
                for (int qq = 0; qq < kTK; ++qq) {
                    float pr[4], dr[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        pr[a] = sm.pt[4 * rg + a][qq];
                        dr[a] = sm.dst[4 * rg + a][qq];
                    }
#pragma unroll
                    for (int t = 0; t < DPT / 4; ++t) {
                        const float4 gg = *reinterpret_cast<const float4*>(&sm.gs[qq][32 * t + 4 * kg]);
                        const float4 q4 = *reinterpret_cast<const float4*>(&sm.qs[qq][32 * t + 4 * kg]);
                        const float gx[4] = {gg.x, gg.y, gg.z, gg.w}, qx[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                        for (int a = 0; a < 4; ++a)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                dva[a][4 * t + e] = fmaf(pr[a], gx[e], dva[a][4 * t + e]);
                                dka[a][4 * t + e] = fmaf(dr[a], qx[e], dka[a][4 * t + e]);
                            }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t u = u0 + 4 * rg + a;
        if (u >= Sb) continue;
#pragma unroll
        for (int t = 0; t < DPT / 4; ++t) {
            const int d0 = 32 * t + 4 * kg;
            if (d0 >= D) continue;
            float x[4], y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[e] = dka[a][4 * t + e] * p.scale;
                y[e] = dva[a][4 * t + e];
            }
            store4_f(dk + (keybase + u) * D + d0, x);
            store4_f(dv + (keybase + u) * D + d0, y);
        }
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

template <typename T, int DMAX>
int launch_tiled_t(const BwdProblem& pr, cudaStream_t stream) {
    const Params P = make_params(pr);
    const unsigned bx = (unsigned)((P.Sb + kTR - 1) / kTR);
    const size_t s1 = sizeof(DqSmem<DMAX>), s2 = sizeof(DkvSmem<DMAX>);
    auto k1 = dq_tiled_kernel<T, DMAX>;
    auto k2 = dkdv_tiled_kernel<T, DMAX>;
    if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2) !=
            cudaSuccess)
        return RA_ERR_CUDA;
    k1<<<dim3(bx, pr.N, pr.B * pr.Hq), kTThreads, s1, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<const T*>(pr.dout), pr.lse, pr.delta, static_cast<T*>(pr.dq), P);
    if (cudaGetLastError() != cudaSuccess) return RA_ERR_CUDA;
    k2<<<dim3(bx, pr.N, pr.B * pr.Hkv), kTThreads, s2, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<const T*>(pr.dout), pr.lse, pr.delta, static_cast<T*>(pr.dk),
        static_cast<T*>(pr.dv), P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

template <typename T>
int launch_simt_d(const BwdProblem& pr, cudaStream_t stream) {
    if (pr.D % 4 == 0) {  // the register-blocked kernels
        if (pr.D <= 32) return launch_tiled_t<T, 32>(pr, stream);
        if (pr.D <= 64) return launch_tiled_t<T, 64>(pr, stream);
        return launch_tiled_t<T, 128>(pr, stream);
    }
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
           p.N <= 65535 && (p.S / p.N + bwd::kTR - 1) / bwd::kTR <= 0x7fffffff;
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
