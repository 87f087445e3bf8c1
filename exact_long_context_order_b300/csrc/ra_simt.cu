// SIMT ring-attention forward kernel: fp32 arithmetic (FFMA, no TF32) for
// float32 or bf16 tensors, any head dimension D <= 256 and any shard size.
//
// It folds exactly like the glossary page's four-device simulation ("Ring
// Attention", "Como funciona a atencao em anel"), with the running maximum
// that page says production kernels subtract: the thread that owns query
// row r of shard i walks the key/value shards j = (i - s) mod N,
// s = 0..N-1, key by key in ascending local order, and keeps a running max m,
// normaliser l and numerator acc[D]; out = acc / l, lse = m + ln l.
// Visibility comes from token positions (contiguous: row p is token p;
// striped: row r of shard j is token r*N + j; zigzag: shard j holds chunk j,
// then chunk 2N-1-j, of 2N chunks of Sb/2 tokens), so masking needs no tiles.
// Key/value rows are staged through shared memory in chunks shared by the
// 128 query rows of a block; chunks past the block's last visible key stop
// the walk of that shard (keys of a shard are in ascending position).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ra.h"

namespace ra {
namespace simt {

constexpr int kRows = 128;

struct Params {
    int B, Hq, Hkv, g, N, D, causal, striped;  // striped: layout 0/1/2
    int64_t S, Sb;
    float scale;
};

// token position of local row r of shard i
__device__ __forceinline__ int64_t token_pos(const Params& p, int64_t i, int64_t r) {
    if (p.striped == 1) return r * p.N + i;
    if (p.striped == 2) {
        const int64_t h = p.Sb / 2;
        return r < h ? i * h + r : (2 * (int64_t)p.N - 1 - i) * h + (r - h);
    }
    return i * p.Sb + r;
}

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T, int DMAX, int KC>
__global__ void __launch_bounds__(kRows) fwd_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                    const T* __restrict__ v, T* __restrict__ out,
                                                    float* __restrict__ lse, const Params p) {
    __shared__ float ks[KC][DMAX];
    __shared__ float vs[KC][DMAX];
    const int i = blockIdx.y;                   // query shard
    const int bh = blockIdx.z;                  // b * Hq + h
    const int b = bh / p.Hq, h = bh % p.Hq;
    const int kvh = h / p.g;
    const int64_t r0 = (int64_t)blockIdx.x * kRows;
    const int64_t r = r0 + threadIdx.x;        // local query row
    const bool active = r < p.Sb;
    const int64_t r_last = (r0 + kRows - 1 < p.Sb) ? r0 + kRows - 1 : p.Sb - 1;
    const int64_t N = p.N;
    const int64_t qpos = token_pos(p, i, r);
    const int64_t qpos_last = token_pos(p, i, r_last);
    const int D = p.D;

    float qr[DMAX], acc[DMAX];
    const T* qrow = q + ((int64_t)bh * p.S + i * p.Sb + (active ? r : 0)) * D;
#pragma unroll
    for (int d = 0; d < DMAX; ++d) {
        qr[d] = (d < D) ? load_f(qrow + d) * p.scale : 0.f;
        acc[d] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const T* kbase = k + ((int64_t)b * p.Hkv + kvh) * p.S * D;
    const T* vbase = v + ((int64_t)b * p.Hkv + kvh) * p.S * D;

    for (int s = 0; s < p.N; ++s) {
        const int j = (int)((i - s + N) % N);
        for (int64_t c0 = 0; c0 < p.Sb; c0 += KC) {
            const int64_t kpos0 = token_pos(p, j, c0);
            if (p.causal && kpos0 > qpos_last) break;
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
                const int64_t c = c0 + kr;
                const int64_t kpos = token_pos(p, j, c);
                if (p.causal && kpos > qpos) continue;
                float sc = 0.f;
#pragma unroll
                for (int d = 0; d < DMAX; ++d) sc = fmaf(qr[d], ks[kr][d], sc);
                if (sc > m) {
                    const float alpha = (m == -INFINITY) ? 0.f : expf(m - sc);
                    l *= alpha;
#pragma unroll
                    for (int d = 0; d < DMAX; ++d) acc[d] *= alpha;
                    m = sc;
                }
                const float pe = expf(sc - m);
                l += pe;
#pragma unroll
                for (int d = 0; d < DMAX; ++d) acc[d] = fmaf(pe, vs[kr][d], acc[d]);
            }
        }
    }
    if (!active) return;
    const int64_t row = (int64_t)bh * p.S + i * p.Sb + r;
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    T* orow = out + row * D;
#pragma unroll
    for (int d = 0; d < DMAX; ++d)
        if (d < D) store_f(orow + d, acc[d] * inv);
    if (lse) lse[row] = (l > 0.f) ? m + logf(l) : -INFINITY;
}

template <typename T, int DMAX>
static int launch_t(const FwdProblem& pr, cudaStream_t stream) {
    Params P;
    P.B = pr.B; P.Hq = pr.Hq; P.Hkv = pr.Hkv; P.g = pr.Hq / pr.Hkv; P.N = pr.N; P.D = pr.D;
    P.causal = pr.causal; P.striped = pr.striped;
    P.S = pr.S; P.Sb = pr.S / pr.N;
    P.scale = pr.scale;
    constexpr int KC = (DMAX <= 64) ? 32 : 16;
    dim3 grid((unsigned)((P.Sb + kRows - 1) / kRows), (unsigned)pr.N, (unsigned)(pr.B * pr.Hq));
    fwd_kernel<T, DMAX, KC><<<grid, kRows, 0, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<T*>(pr.out), pr.lse, P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

template <typename T>
static int launch_d(const FwdProblem& pr, cudaStream_t stream) {
    if (pr.D <= 32) return launch_t<T, 32>(pr, stream);
    if (pr.D <= 64) return launch_t<T, 64>(pr, stream);
    if (pr.D <= 128) return launch_t<T, 128>(pr, stream);
    return launch_t<T, 256>(pr, stream);
}

}  // namespace simt

bool simt_supported(const FwdProblem& p) {
    // grid (row blocks, N, B*Hq): y and z are limited to 65535
    return p.D <= 256 && (int64_t)p.B * p.Hq <= 65535 && p.N <= 65535 &&
           (p.S / p.N + 127) / 128 <= 0x7fffffff;
}

int launch_simt(const FwdProblem& p, unsigned int* /*status*/, cudaStream_t stream) {
    if (!simt_supported(p)) return RA_ERR_UNSUPPORTED;
    return p.dtype == RA_F32 ? simt::launch_d<float>(p, stream)
                             : simt::launch_d<__nv_bfloat16>(p, stream);
}

}  // namespace ra
