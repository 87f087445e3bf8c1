// ra_forward_noalloc: the bf16 tensor-core forward for callers that must not
// allocate device memory.
//
// Some programs cannot call cudaMalloc at the time they run attention: a
// serving process that has handed the whole GPU to its own memory pool up
// front, a framework whose caching allocator owns every byte of device memory,
// or latency-critical code that cannot accept cudaMalloc's implicit device
// synchronisation or its failure when memory is exhausted.  ra_forward
// allocates a small scratch block on its first tensor-core call on a device;
// this entry point instead keeps its scratch (the kernel's work-queue counter)
// in a file-scope static __device__ array that exists as soon as the module is
// loaded, so nothing is ever allocated.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ra.h"

namespace {

// Scratch of ra_forward_noalloc: 256 bytes on every device that loads the
// library, held until the process exits.  Word 0 is the work-queue counter of
// the running call.  Every call uses the same array, so calls whose kernels
// overlap on the GPU race on it.
constexpr int kNoAllocScratchWords = 64;
constexpr int64_t kNoAllocScratchBytes = kNoAllocScratchWords * 4;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Device address of g_noalloc_scratch, resolved once per device.  In host code
// the array's name only stands in for the symbol; it is not a device address.
unsigned int* g_scratch_addr[kMaxDevices];

int scratch_address(int dev, unsigned int** addr) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            ra::note_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return RA_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<unsigned int*>(p);
    }
    *addr = g_scratch_addr[dev];
    return RA_OK;
}

}  // namespace

extern "C" int ra_forward_noalloc(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int Hq, int Hkv, int64_t S, int D, int N,
                                  int causal, int striped, float scale, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || D <= 0 || N <= 0) return RA_ERR_INVALID_ARG;
    if (S % N != 0 || Hq % Hkv != 0) return RA_ERR_INVALID_ARG;
    if (striped < RA_LAYOUT_CONTIGUOUS || striped > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    if (B == 0 || S == 0) return RA_OK;  // empty: nothing is read or written
    if (!q || !k || !v || !out) return RA_ERR_INVALID_ARG;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
                          reinterpret_cast<uintptr_t>(lse);
    if (mis & 15u) return RA_ERR_ALIGN;

    ra::FwdProblem p;
    p.q = q; p.k = k; p.v = v; p.out = out; p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.S = S; p.D = D; p.N = N;
    p.causal = causal ? 1 : 0;
    p.striped = striped;
    p.scale = (scale > 0.f && std::isfinite(scale)) ? scale : (float)(1.0 / std::sqrt((double)D));
    p.dtype = RA_BF16;
    if (!ra::tc_supported(p)) return RA_ERR_UNSUPPORTED;

    // The scratch this call needs must fit the static array: one 32-bit work
    // counter, and the work-item count must fit that counter.
    const int64_t need_bytes = 4;
    const int64_t Sb = S / N;
    const int64_t items_bound = (int64_t)B * Hq * N * ((Sb + 127) / 128);  // >= work items
    if (need_bytes > kNoAllocScratchBytes || items_bound >= (int64_t)1 << 31)
        return RA_ERR_CAPACITY;

    // status word, SM count and architecture (sm_103 only), resolved once per device
    unsigned int* status = nullptr;
    int sms = 0;
    int rc = ra::device_info(&status, &sms);
    if (rc) return rc;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        ra::note_cuda_error(e);
        return RA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    unsigned int* scratch = nullptr;
    if ((rc = scratch_address(dev, &scratch))) return rc;
    // launch_tc zeroes the counter on `stream` before the kernel starts, so the
    // previous call's final count never leaks into this one.
    rc = ra::launch_tc(p, nullptr, status, scratch, sms, static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) ra::note_cuda_error(cudaGetLastError());
    return rc;
}
