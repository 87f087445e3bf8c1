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
// Two kernels: for D % 4 == 0 and D <= 128 a register-blocked one (64 query
// rows per block, 4x4 scores and a 4-row slice of the numerator per thread);
// otherwise one thread per query row holding the row's q and numerator.  Both
// stage key/value rows through shared memory in chunks shared by the block's
// query rows; chunks past the block's last visible key stop the walk of that
// shard (keys of a shard are in ascending position).
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

// ---------------------------------------------------------------- tiled kernel (D <= 128)
// The same fold with register blocking: a block takes 64 query rows of one
// (b, h, shard) and walks the key shards in ring order in chunks of 32 keys
// staged in shared memory.  Thread (rg, kg) = (tid / 8, tid % 8) computes the
// scores of rows 4rg..4rg+3 against keys 4kg..4kg+3 of the chunk, and owns
// the numerator of the same rows on dims {32t + 4kg + i}.  The running max and
// normaliser of a row are kept by the eight threads of its row group, which
// reduce a chunk's row max and row sum with shuffles over the lane bits that
// hold kg.  Needs D % 4 == 0 (rows are moved four elements at a time).
constexpr int kTR = 64;       // query rows per block
constexpr int kTK = 32;       // keys per chunk
constexpr int kTThreads = 128;

template <int DMAX>
struct TiledSmem {
    float qt[DMAX][kTR];      // scale * q, transposed; rows past the shard are 0
    float kt[DMAX][kTK];      // k of the chunk, transposed
    float vs[kTK][DMAX];      // v of the chunk
    float ps[kTR][kTK + 1];   // P of the chunk
};

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

template <typename T, int DMAX>
__global__ void __launch_bounds__(kTThreads)
    fwd_tiled_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     T* __restrict__ out, float* __restrict__ lse, const Params p) {
    constexpr int DPT = DMAX / 8;  // numerator dims per thread
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TiledSmem<DMAX>& sm = *reinterpret_cast<TiledSmem<DMAX>*>(smem_raw);
    const int tid = threadIdx.x, rg = tid >> 3, kg = tid & 7;
    const int i = blockIdx.y;   // query shard
    const int bh = blockIdx.z;  // b * Hq + h
    const int b = bh / p.Hq, h = bh % p.Hq, kvh = h / p.g;
    const int64_t r0 = (int64_t)blockIdx.x * kTR;
    const int64_t N = p.N, Sb = p.Sb;
    const int D = p.D;
    const int64_t r_last = (r0 + kTR - 1 < Sb) ? r0 + kTR - 1 : Sb - 1;
    const int64_t qpos_last = token_pos(p, i, r_last);
    int64_t qpos[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) qpos[a] = token_pos(p, i, r0 + 4 * rg + a);

    // q tile, transposed and scaled: lanes take consecutive rows
    const T* qbase = q + ((int64_t)bh * p.S + i * Sb) * D;
    for (int e = tid; e < kTR * (DMAX / 4); e += kTThreads) {
        const int r = e % kTR, d4 = e / kTR;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (r0 + r < Sb && 4 * d4 < D) load4_f(qbase + (r0 + r) * D + 4 * d4, x);
#pragma unroll
        for (int a = 0; a < 4; ++a) sm.qt[4 * d4 + a][r] = x[a] * p.scale;
    }
    float o[4][DPT];
    float m[4], l[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        m[a] = -INFINITY;
        l[a] = 0.f;
#pragma unroll
        for (int d = 0; d < DPT; ++d) o[a][d] = 0.f;
    }
    const T* kbase = k + ((int64_t)b * p.Hkv + kvh) * p.S * D;
    const T* vbase = v + ((int64_t)b * p.Hkv + kvh) * p.S * D;

    for (int s = 0; s < p.N; ++s) {
        const int j = (int)((i - s + N) % N);
        for (int64_t c0 = 0; c0 < Sb; c0 += kTK) {
            if (p.causal && token_pos(p, j, c0) > qpos_last) break;  // keys ascend in a shard
            const int nk = (int)((Sb - c0 < kTK) ? Sb - c0 : kTK);
            const T* kc = kbase + (j * Sb + c0) * D;
            const T* vc = vbase + (j * Sb + c0) * D;
            __syncthreads();  // the previous chunk's reads are done
            // k transposed: lanes take consecutive keys (conflict-free stores)
            for (int e = tid; e < kTK * (DMAX / 4); e += kTThreads) {
                const int key = e % kTK, d4 = e / kTK;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (key < nk && 4 * d4 < D) load4_f(kc + (int64_t)key * D + 4 * d4, x);
#pragma unroll
                for (int a = 0; a < 4; ++a) sm.kt[4 * d4 + a][key] = x[a];
            }
            // v as is: lanes take consecutive dims (coalesced)
            for (int e = tid; e < kTK * (DMAX / 4); e += kTThreads) {
                const int d4 = e % (DMAX / 4), key = e / (DMAX / 4);
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (key < nk && 4 * d4 < D) load4_f(vc + (int64_t)key * D + 4 * d4, x);
                store4_f(&sm.vs[key][4 * d4], x);
            }
            __syncthreads();
            // scores of rows 4rg.. against keys 4kg..
            float sc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[a][c] = 0.f;
#pragma unroll 8
            for (int d = 0; d < DMAX; ++d) {
                const float4 qa = *reinterpret_cast<const float4*>(&sm.qt[d][4 * rg]);
                const float4 kb = *reinterpret_cast<const float4*>(&sm.kt[d][4 * kg]);
                const float qv[4] = {qa.x, qa.y, qa.z, qa.w}, kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c) sc[a][c] = fmaf(qv[a], kv[c], sc[a][c]);
            }
            // visibility from positions; keys past the shard are invisible
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = 4 * kg + c;
                const int64_t kpos = token_pos(p, j, c0 + key);
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    if (key >= nk || (p.causal && kpos > qpos[a])) sc[a][c] = -INFINITY;
            }
            // online softmax over the chunk, per row of the group
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                float mx = fmaxf(fmaxf(sc[a][0], sc[a][1]), fmaxf(sc[a][2], sc[a][3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                const float mn = fmaxf(m[a], mx);
                float alpha = 1.f, rs = 0.f;
                if (mn != -INFINITY) {
                    alpha = (m[a] == -INFINITY) ? 0.f : expf(m[a] - mn);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        sc[a][c] = (sc[a][c] == -INFINITY) ? 0.f : expf(sc[a][c] - mn);
                        rs += sc[a][c];
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) sc[a][c] = 0.f;
                }
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                rs += __shfl_xor_sync(0xffffffffu, rs, 4);
                l[a] = l[a] * alpha + rs;
                m[a] = mn;
#pragma unroll
                for (int d = 0; d < DPT; ++d) o[a][d] *= alpha;
#pragma unroll
                for (int c = 0; c < 4; ++c) sm.ps[4 * rg + a][4 * kg + c] = sc[a][c];
            }
            __syncthreads();
            // numerator += P v on dims {32t + 4kg + e}
#pragma unroll 4
            for (int key = 0; key < kTK; ++key) {
                float pr[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) pr[a] = sm.ps[4 * rg + a][key];
#pragma unroll
                for (int t = 0; t < DPT / 4; ++t) {
                    const float4 vv = *reinterpret_cast<const float4*>(&sm.vs[key][32 * t + 4 * kg]);
                    const float vx[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[a][4 * t + e] = fmaf(pr[a], vx[e], o[a][4 * t + e]);
                }
            }
        }
    }
    // epilogue: out = numerator / l, lse = m + ln l
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t r = r0 + 4 * rg + a;
        if (r >= Sb) continue;
        const int64_t row = (int64_t)bh * p.S + i * Sb + r;
        const float inv = (l[a] > 0.f) ? 1.f / l[a] : 0.f;
#pragma unroll
        for (int t = 0; t < DPT / 4; ++t) {
            const int d0 = 32 * t + 4 * kg;
            if (d0 >= D) continue;
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = o[a][4 * t + e] * inv;
            store4_f(out + row * D + d0, x);
        }
        if (lse && kg == 0) lse[row] = (l[a] > 0.f) ? m[a] + logf(l[a]) : -INFINITY;
    }
}

template <typename T, int DMAX>
static int launch_tiled(const FwdProblem& pr, cudaStream_t stream) {
    Params P;
    P.B = pr.B; P.Hq = pr.Hq; P.Hkv = pr.Hkv; P.g = pr.Hq / pr.Hkv; P.N = pr.N; P.D = pr.D;
    P.causal = pr.causal; P.striped = pr.striped;
    P.S = pr.S; P.Sb = pr.S / pr.N;
    P.scale = pr.scale;
    const size_t smem = sizeof(TiledSmem<DMAX>);
    auto kern = fwd_tiled_kernel<T, DMAX>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return RA_ERR_CUDA;
    dim3 grid((unsigned)((P.Sb + kTR - 1) / kTR), (unsigned)pr.N, (unsigned)(pr.B * pr.Hq));
    kern<<<grid, kTThreads, smem, stream>>>(
        static_cast<const T*>(pr.q), static_cast<const T*>(pr.k), static_cast<const T*>(pr.v),
        static_cast<T*>(pr.out), pr.lse, P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
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
    if (pr.D % 4 == 0 && pr.D <= 128) {  // the register-blocked kernel
        if (pr.D <= 32) return launch_tiled<T, 32>(pr, stream);
        if (pr.D <= 64) return launch_tiled<T, 64>(pr, stream);
        return launch_tiled<T, 128>(pr, stream);
    }
    if (pr.D <= 32) return launch_t<T, 32>(pr, stream);
    if (pr.D <= 64) return launch_t<T, 64>(pr, stream);
    if (pr.D <= 128) return launch_t<T, 128>(pr, stream);
    return launch_t<T, 256>(pr, stream);
}

}  // namespace simt

bool simt_supported(const FwdProblem& p) {
    // grid (row blocks, N, B*Hq): y and z are limited to 65535
    return p.D <= 256 && (int64_t)p.B * p.Hq <= 65535 && p.N <= 65535 &&
           (p.S / p.N + simt::kTR - 1) / simt::kTR <= 0x7fffffff;
}

int launch_simt(const FwdProblem& p, unsigned int* /*status*/, cudaStream_t stream) {
    if (!simt_supported(p)) return RA_ERR_UNSUPPORTED;
    return p.dtype == RA_F32 ? simt::launch_d<float>(p, stream)
                             : simt::launch_d<__nv_bfloat16>(p, stream);
}

}  // namespace ra
