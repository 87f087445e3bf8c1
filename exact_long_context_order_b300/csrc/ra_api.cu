// C ABI of the ring-attention library: argument validation, the per-device
// status word, kernel dispatch and the host-side fold planner.  Every entry
// point returns an RA_* status and never throws.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ra.h"
#include "schedule.cuh"

namespace {

// One status word per device, set by kernels (bounded waits that ran out,
// bounds checks) and read/cleared by ra_check.
__device__ unsigned int g_ra_status;

constexpr int kMaxDevices = 64;
// Work counters of the tensor-core kernel: one small block per device,
// allocated on first use, holding kWorkSlots counters; each launch takes the
// next slot (zeroed on its stream), so up to kWorkSlots launches may be in
// flight on one device at once.
constexpr int kWorkSlots = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices];
unsigned int* g_work[kMaxDevices];
unsigned int g_work_next[kMaxDevices];
int g_sm_count[kMaxDevices];
int g_arch_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
thread_local char g_cuda_msg[256] = "";

void note_cuda(cudaError_t e) {
    snprintf(g_cuda_msg, sizeof(g_cuda_msg), "%s", cudaGetErrorString(e));
}

// Resolves this device's status word address, SM count and architecture.
int device_state(unsigned int** status, int* sm_count) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { note_cuda(e); return RA_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
            note_cuda(e);
            return RA_ERR_CUDA;
        }
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch_ok[dev] != 1) return RA_ERR_UNSUPPORTED;
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_ra_status)) != cudaSuccess) { note_cuda(e); return RA_ERR_CUDA; }
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    if (status) *status = g_status_ptr[dev];
    if (sm_count) *sm_count = g_sm_count[dev];
    return RA_OK;
}

// Next work-counter slot of the current device (allocates the block once).
int work_slot(unsigned int** slot) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { note_cuda(e); return RA_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_work[dev]) {
        void* p = nullptr;
        if ((e = cudaMalloc(&p, kWorkSlots * 64)) != cudaSuccess) { note_cuda(e); return RA_ERR_CUDA; }
        g_work[dev] = static_cast<unsigned int*>(p);
    }
    // 64-byte spacing keeps concurrent launches' counters on separate lines
    *slot = g_work[dev] + (g_work_next[dev]++ % kWorkSlots) * 16;
    return RA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// An empty problem (no batch entry or no token) is valid; nothing is read or
// written, so its buffer pointers are not checked.
bool empty_problem(int B, int64_t S) { return B == 0 || S == 0; }

int validate_forward(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, int B, int Hq, int Hkv, int64_t S, int D, int N, int dtype,
                     int layout) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || S < 0 || D <= 0 || N <= 0) return RA_ERR_INVALID_ARG;
    if (S % N != 0 || Hq % Hkv != 0) return RA_ERR_INVALID_ARG;
    if (layout < RA_LAYOUT_CONTIGUOUS || layout > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    if (layout == RA_LAYOUT_ZIGZAG && (S / N) % 2) return RA_ERR_INVALID_ARG;
    if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_INVALID_ARG;
    if (D > 256) return RA_ERR_UNSUPPORTED;
    if (empty_problem(B, S)) return RA_OK;
    if (!q || !k || !v || !out) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_ALIGN;
    if (lse && !aligned16(lse)) return RA_ERR_ALIGN;
    return RA_OK;
}

ra::FwdProblem make_problem(const void* q, const void* k, const void* v, void* out, float* lse,
                            int B, int Hq, int Hkv, int64_t S, int D, int N, int causal,
                            int striped, float scale, int dtype) {
    ra::FwdProblem p;
    p.q = q; p.k = k; p.v = v; p.out = out; p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.S = S; p.D = D; p.N = N;
    p.causal = causal ? 1 : 0;
    p.striped = striped;
    p.scale = (scale > 0.f && std::isfinite(scale)) ? scale : (float)(1.0 / std::sqrt((double)D));
    p.dtype = dtype;
    return p;
}

// Workspace of ra_backward: delta, float32 per query row, padded to 256
// bytes.  -1 when the size overflows.
int64_t backward_workspace_bytes(int B, int Hq, int64_t S, int D) {
    (void)D;
    const double est = 4.0 * B * Hq * (double)S + 256;
    if (est > 4.0e18) return -1;
    return ((4 * (int64_t)B * Hq * S) + 255) / 256 * 256;
}

// Validates ra_backward's arguments on the host and fills the problem
// (everything but the kernel choice).  Returns RA_OK or the error code.
int prepare_backward(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     void* workspace, int64_t workspace_bytes, int B, int Hq, int Hkv, int64_t S,
                     int D, int N, int causal, int striped, float scale, int dtype,
                     ra::BwdProblem* p) {
    int rc = validate_forward(q, k, v, out, nullptr, B, Hq, Hkv, S, D, N, dtype, striped);
    if (rc) return rc;
    if (D > 128) return RA_ERR_UNSUPPORTED;
    p->B = B; p->S = S;
    if (empty_problem(B, S)) return RA_OK;
    if (!lse || !dout || !dq || !dk || !dv || !workspace) return RA_ERR_INVALID_ARG;
    if (!aligned16(lse) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv) || !aligned16(workspace))
        return RA_ERR_ALIGN;
    const int64_t need = backward_workspace_bytes(B, Hq, S, D);
    if (need < 0) return RA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return RA_ERR_CAPACITY;
    p->q = q; p->k = k; p->v = v; p->out = out; p->lse = lse; p->dout = dout;
    p->dq = dq; p->dk = dk; p->dv = dv;
    p->delta = static_cast<float*>(workspace);
    p->B = B; p->Hq = Hq; p->Hkv = Hkv; p->S = S; p->D = D; p->N = N;
    p->causal = causal ? 1 : 0;
    p->striped = striped;
    p->scale = (scale > 0.f && std::isfinite(scale)) ? scale : (float)(1.0 / std::sqrt((double)D));
    p->dtype = dtype;
    return RA_OK;
}

// ra_forward_host's pipeline: per device, a host-to-device copy stream, a
// device-to-host copy stream, two compute streams and the events that order
// them.  Created on first use and kept for the life of the process.  The
// enqueue sequence of one call holds g_pipe_mu, because every call re-records
// the same events.
constexpr int kHostChunks = 8;
struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr, comp[2] = {nullptr, nullptr};
    cudaEvent_t fork = nullptr, join = nullptr, in[kHostChunks] = {}, done[kHostChunks] = {};
    // one event per side stream, recorded only when a call fails part-way
    cudaEvent_t unwind[4] = {};
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDevices];

// The current device's pipeline; the caller holds g_pipe_mu.
int host_pipe(HostPipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { note_cuda(e); return RA_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    HostPipe& hp = g_pipe[dev];
    if (!hp.ready) {
        const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
        cudaStream_t* streams[4] = {&hp.h2d, &hp.d2h, &hp.comp[0], &hp.comp[1]};
        for (cudaStream_t* st : streams)
            if (!*st && (e = cudaStreamCreateWithFlags(st, sf)) != cudaSuccess) {
                note_cuda(e);
                return RA_ERR_CUDA;
            }
        cudaEvent_t* events[6 + 2 * kHostChunks];
        int n = 0;
        events[n++] = &hp.fork;
        events[n++] = &hp.join;
        for (cudaEvent_t& u : hp.unwind) events[n++] = &u;
        for (int c = 0; c < kHostChunks; ++c) {
            events[n++] = &hp.in[c];
            events[n++] = &hp.done[c];
        }
        for (int j = 0; j < n; ++j)
            if (!*events[j] && (e = cudaEventCreateWithFlags(events[j], ef)) != cudaSuccess) {
                note_cuda(e);
                return RA_ERR_CUDA;
            }
        hp.ready = true;
    }
    *out = &hp;
    return RA_OK;
}

}  // namespace

int ra::device_status_word(unsigned int** status) { return device_state(status, nullptr); }
int ra::device_info(unsigned int** status, int* sm_count) { return device_state(status, sm_count); }
void ra::note_cuda_error(cudaError_t e) { note_cuda(e); }

extern "C" {

int ra_forward_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                  int Hq, int Hkv, int64_t S, int D, int N, int causal, int striped, float scale,
                  int dtype, int kernel, void* stream) {
    int rc = validate_forward(q, k, v, out, lse, B, Hq, Hkv, S, D, N, dtype, striped);
    if (rc) return rc;
    if (kernel != RA_KERNEL_AUTO && kernel != RA_KERNEL_TC && kernel != RA_KERNEL_SIMT)
        return RA_ERR_INVALID_ARG;
    if (empty_problem(B, S)) return RA_OK;
    const ra::FwdProblem p = make_problem(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped,
                                          scale, dtype);
    // the kernels' envelopes are host checks, made before any CUDA call
    const bool tc_ok = ra::tc_supported(p);
    if (kernel == RA_KERNEL_TC && !tc_ok) return RA_ERR_UNSUPPORTED;
    const bool use_tc = kernel == RA_KERNEL_TC || (kernel == RA_KERNEL_AUTO && tc_ok);
    if (!use_tc && !ra::simt_supported(p)) return RA_ERR_UNSUPPORTED;
    unsigned int* status = nullptr;
    int sms = 0;
    if ((rc = device_state(&status, &sms))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_tc) {
        unsigned int* work = nullptr;
        if ((rc = work_slot(&work))) return rc;
        rc = ra::launch_tc(p, nullptr, status, work, sms, st, 0, 0,
                           kernel == RA_KERNEL_AUTO ? 1 : 0);
    } else
        rc = ra::launch_simt(p, status, st);
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_forward(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
               int Hkv, int64_t S, int D, int N, int causal, int striped, float scale, int dtype,
               void* stream) {
    return ra_forward_ex(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped, scale, dtype,
                         RA_KERNEL_AUTO, stream);
}

int ra_backward_workspace(int B, int Hq, int64_t S, int D, int64_t* bytes) {
    if (!bytes || B < 0 || Hq <= 0 || S < 0 || D <= 0) return RA_ERR_INVALID_ARG;
    const int64_t wb = backward_workspace_bytes(B, Hq, S, D);
    if (wb < 0) return RA_ERR_INVALID_ARG;
    *bytes = wb;
    return RA_OK;
}

int ra_backward_ex(const void* q, const void* k, const void* v, const void* out,
                   const float* lse, const void* dout, void* dq, void* dk, void* dv,
                   void* workspace, int64_t workspace_bytes, int B, int Hq, int Hkv, int64_t S,
                   int D, int N, int causal, int striped, float scale, int dtype, int kernel,
                   void* stream) {
    if (kernel != RA_KERNEL_AUTO && kernel != RA_KERNEL_TC && kernel != RA_KERNEL_SIMT)
        return RA_ERR_INVALID_ARG;
    ra::BwdProblem p;
    int rc = prepare_backward(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B,
                              Hq, Hkv, S, D, N, causal, striped, scale, dtype, &p);
    if (rc) return rc;
    if (empty_problem(B, S)) return RA_OK;
    // the kernels' envelopes are host checks, made before any CUDA call
    const bool tc_ok = ra::tc_bwd_supported(p);
    if (kernel == RA_KERNEL_TC && !tc_ok) return RA_ERR_UNSUPPORTED;
    const bool use_tc = kernel == RA_KERNEL_TC || (kernel == RA_KERNEL_AUTO && tc_ok);
    if (!ra::bwd_delta_supported(p) || (!use_tc && !ra::simt_bwd_supported(p)))
        return RA_ERR_UNSUPPORTED;
    unsigned int* status = nullptr;
    int sms = 0;
    if ((rc = device_state(&status, &sms))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = ra::launch_bwd_delta(p, st))) {
        if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
        return rc;
    }
    if (use_tc) {
        unsigned int* work = nullptr;
        if ((rc = work_slot(&work))) return rc;
        rc = ra::launch_bwd_tc(p, status, work, sms, st);
    } else
        rc = ra::launch_bwd_simt(p, st);
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_watchdog_selftest_backward(const void* q, const void* k, const void* v, const void* out,
                                  const float* lse, const void* dout, void* dq, void* dk,
                                  void* dv, void* workspace, int64_t workspace_bytes, int B,
                                  int Hq, int Hkv, int64_t S, int D, int N, int causal,
                                  int striped, float scale, int64_t timeout_cycles, int which,
                                  void* stream) {
    if (timeout_cycles < 100000 || timeout_cycles > 4000000000ll) return RA_ERR_INVALID_ARG;
    if (which != 0 && which != 1) return RA_ERR_INVALID_ARG;
    ra::BwdProblem p;
    int rc = prepare_backward(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B,
                              Hq, Hkv, S, D, N, causal, striped, scale, RA_BF16, &p);
    if (rc) return rc;
    if (empty_problem(B, S)) return RA_ERR_INVALID_ARG;  // the self test needs a kernel to run
    if (!ra::tc_bwd_supported(p)) return RA_ERR_UNSUPPORTED;
    unsigned int* status = nullptr;
    int sms = 0;
    if ((rc = device_state(&status, &sms))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = ra::launch_bwd_delta(p, st))) {
        if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
        return rc;
    }
    unsigned int* work = nullptr;
    if ((rc = work_slot(&work))) return rc;
    rc = ra::launch_bwd_tc_selftest(p, status, work, sms, st, timeout_cycles, which);
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_backward(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, void* workspace,
                int64_t workspace_bytes, int B, int Hq, int Hkv, int64_t S, int D, int N,
                int causal, int striped, float scale, int dtype, void* stream) {
    return ra_backward_ex(q, k, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, Hq,
                          Hkv, S, D, N, causal, striped, scale, dtype, RA_KERNEL_AUTO, stream);
}

int ra_forward_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                    float* lse_host, void* q_dev, void* k_dev, void* v_dev, void* out_dev,
                    float* lse_dev, int B, int Hq, int Hkv, int64_t S, int D, int N, int causal,
                    int striped, float scale, int dtype, void* stream) {
    if ((lse_host != nullptr) != (lse_dev != nullptr)) return RA_ERR_INVALID_ARG;
    int rc = validate_forward(q_dev, k_dev, v_dev, out_dev, lse_dev, B, Hq, Hkv, S, D, N, dtype,
                              striped);
    if (rc) return rc;
    if (empty_problem(B, S)) return RA_OK;
    if (!q_host || !k_host || !v_host || !out_host) return RA_ERR_INVALID_ARG;
    const int64_t esz = (dtype == RA_F32) ? 4 : 2;
    const int64_t G = (int64_t)B * Hkv;  // (batch, KV head) groups
    int nch = (G >= 4 && G <= 0x7fffffff) ? (int)std::min<int64_t>(G, kHostChunks) : 1;
    {
        // A problem ra_forward runs as stream-K cuts items at places a chunk
        // would not: run it whole, so the outputs stay the same bits.
        int sms = 0;
        if ((rc = device_state(nullptr, &sms))) return rc;
        const ra::FwdProblem whole = make_problem(q_dev, k_dev, v_dev, out_dev, lse_dev, B, Hq,
                                                  Hkv, S, D, N, causal, striped, scale, dtype);
        if (ra::tc_uses_streamk(whole, sms)) nch = 1;
    }
    const int g = Hq / Hkv;
    const int64_t qg = (int64_t)g * S * D * esz, kvg = S * D * esz, lg = (int64_t)g * S;
    // Every chunk is a sub-problem whose device pointers must meet ra_forward's
    // 16-byte rule; if one chunk's offset would not, run the call in order.
    for (int c = 1; c < nch; ++c) {
        const int64_t g0 = G * c / nch;
        if ((g0 * qg) % 16 || (g0 * kvg) % 16 || (lse_dev && (g0 * lg * 4) % 16)) {
            nch = 1;
            break;
        }
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    auto fail = [](cudaError_t err) {
        note_cuda(err);
        return RA_ERR_CUDA;
    };
    if (nch == 1) {  // too few groups to pipeline: everything in order on the caller's stream
        const int64_t qbytes = (int64_t)B * Hq * S * D * esz, kvbytes = G * S * D * esz;
        if ((e = cudaMemcpyAsync(q_dev, q_host, qbytes, cudaMemcpyHostToDevice, st)) ||
            (e = cudaMemcpyAsync(k_dev, k_host, kvbytes, cudaMemcpyHostToDevice, st)) ||
            (e = cudaMemcpyAsync(v_dev, v_host, kvbytes, cudaMemcpyHostToDevice, st)))
            return fail(e);
        if ((rc = ra_forward_ex(q_dev, k_dev, v_dev, out_dev, lse_dev, B, Hq, Hkv, S, D, N, causal,
                                striped, scale, dtype, RA_KERNEL_AUTO, stream)))
            return rc;
        if ((e = cudaMemcpyAsync(out_host, out_dev, qbytes, cudaMemcpyDeviceToHost, st)))
            return fail(e);
        if (lse_host && (e = cudaMemcpyAsync(lse_host, lse_dev, (int64_t)B * Hq * S * 4,
                                             cudaMemcpyDeviceToHost, st)))
            return fail(e);
        return RA_OK;
    }
    // Pipelined over chunks of consecutive (batch, KV head) groups.  A group's
    // q heads, k, v, out and lse rows are contiguous, so a chunk is itself a
    // problem (B' = its groups, Hq' = Hq / Hkv, Hkv' = 1) and the same kernels
    // compute the same bits for it.  Chunk c's copies in run on the h2d
    // stream, its forward on compute stream c % 2 (so a chunk's kernel can
    // start on the SMs that the previous chunk's tail frees), its copies out
    // on the d2h stream; all three are forked from and joined back to the
    // caller's stream.
    const ra::FwdProblem full = make_problem(q_dev, k_dev, v_dev, out_dev, lse_dev, B, Hq, Hkv, S,
                                             D, N, causal, striped, scale, dtype);
    if (!ra::tc_supported(full) && !ra::simt_supported(full)) return RA_ERR_UNSUPPORTED;
    if ((rc = device_state(nullptr, nullptr))) return rc;
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe* hp = nullptr;
    if ((rc = host_pipe(&hp))) return rc;
    if ((e = cudaEventRecord(hp->fork, st))) return fail(e);
    const cudaStream_t side[4] = {hp->h2d, hp->d2h, hp->comp[0], hp->comp[1]};
    for (int x = 0; x < 4; ++x)
        if ((e = cudaStreamWaitEvent(side[x], hp->fork, 0))) {
            // the streams forked so far hold no work yet; join them anyway
            for (int y = 0; y < x; ++y)
                if (cudaEventRecord(hp->unwind[y], side[y]) == cudaSuccess)
                    cudaStreamWaitEvent(st, hp->unwind[y], 0);
            return fail(e);
        }
    // After the fork, a failure part-way must still make the caller's stream
    // wait for whatever was enqueued on the side streams (copies and kernels
    // that use the caller's buffers), so `stream` keeps ordering the call.
    auto unwind = [&](int code) {
        for (int y = 0; y < 4; ++y)
            if (cudaEventRecord(hp->unwind[y], side[y]) == cudaSuccess)
                cudaStreamWaitEvent(st, hp->unwind[y], 0);
        return code;
    };
    auto fail_joined = [&](cudaError_t err) {
        note_cuda(err);
        return unwind(RA_ERR_CUDA);
    };
    char* qd = static_cast<char*>(q_dev);
    char* kd = static_cast<char*>(k_dev);
    char* vd = static_cast<char*>(v_dev);
    char* od = static_cast<char*>(out_dev);
    const char* qh = static_cast<const char*>(q_host);
    const char* kh = static_cast<const char*>(k_host);
    const char* vh = static_cast<const char*>(v_host);
    char* oh = static_cast<char*>(out_host);
    for (int c = 0; c < nch; ++c) {
        const int64_t g0 = G * c / nch, m = G * (c + 1) / nch - g0;
        if ((e = cudaMemcpyAsync(qd + g0 * qg, qh + g0 * qg, m * qg, cudaMemcpyHostToDevice,
                                 hp->h2d)) ||
            (e = cudaMemcpyAsync(kd + g0 * kvg, kh + g0 * kvg, m * kvg, cudaMemcpyHostToDevice,
                                 hp->h2d)) ||
            (e = cudaMemcpyAsync(vd + g0 * kvg, vh + g0 * kvg, m * kvg, cudaMemcpyHostToDevice,
                                 hp->h2d)) ||
            (e = cudaEventRecord(hp->in[c], hp->h2d)))
            return fail_joined(e);
        cudaStream_t cs = hp->comp[c & 1];
        if ((e = cudaStreamWaitEvent(cs, hp->in[c], 0))) return fail_joined(e);
        if ((rc = ra_forward_ex(qd + g0 * qg, kd + g0 * kvg, vd + g0 * kvg, od + g0 * qg,
                                lse_dev ? lse_dev + g0 * lg : nullptr, (int)m, g, 1, S, D, N,
                                causal, striped, scale, dtype, RA_KERNEL_AUTO, cs)))
            return unwind(rc);
        if ((e = cudaEventRecord(hp->done[c], cs)) ||
            (e = cudaStreamWaitEvent(hp->d2h, hp->done[c], 0)) ||
            (e = cudaMemcpyAsync(oh + g0 * qg, od + g0 * qg, m * qg, cudaMemcpyDeviceToHost,
                                 hp->d2h)))
            return fail_joined(e);
        if (lse_host && (e = cudaMemcpyAsync(lse_host + g0 * lg, lse_dev + g0 * lg, m * lg * 4,
                                             cudaMemcpyDeviceToHost, hp->d2h)))
            return fail_joined(e);
    }
    // every compute launch precedes a copy out, so the d2h stream's end joins all
    if ((e = cudaEventRecord(hp->join, hp->d2h)) || (e = cudaStreamWaitEvent(st, hp->join, 0)))
        return fail_joined(e);
    return RA_OK;
}

int ra_fold_log(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                int Hkv, int64_t S, int D, int N, int causal, int striped, float scale,
                int32_t* log, int32_t* counts, int max_entries, void* stream) {
    int rc = validate_forward(q, k, v, out, lse, B, Hq, Hkv, S, D, N, RA_BF16, striped);
    if (rc) return rc;
    if (empty_problem(B, S)) return RA_ERR_INVALID_ARG;  // nothing to log
    if (!log || !counts || !aligned16(log) || ((uintptr_t)counts & 3u)) return RA_ERR_INVALID_ARG;
    const ra::FwdProblem p = make_problem(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped,
                                          scale, RA_BF16);
    if (!ra::tc_supported(p)) return RA_ERR_UNSUPPORTED;
    if ((int64_t)max_entries < (int64_t)N * ((S / N + 127) / 128)) return RA_ERR_CAPACITY;
    unsigned int* status = nullptr;
    int sms = 0;
    if ((rc = device_state(&status, &sms))) return rc;
    ra::FoldLog fl{log, counts, max_entries};
    unsigned int* work = nullptr;
    if ((rc = work_slot(&work))) return rc;
    rc = ra::launch_tc(p, &fl, status, work, sms, static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_ring_step(const void* q, const void* k, const void* v, float* state_o, float* state_lse,
                 void* out, float* lse, int B, int Hq, int Hkv, int64_t Sb, int D, int N, int i,
                 int j, int causal, int layout, float scale, int flags, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sb < 0 || D <= 0 || N <= 0) return RA_ERR_INVALID_ARG;
    if (Hq % Hkv || i < 0 || i >= N || j < 0 || j >= N) return RA_ERR_INVALID_ARG;
    if (layout < RA_LAYOUT_CONTIGUOUS || layout > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    if (layout == RA_LAYOUT_ZIGZAG && Sb % 2) return RA_ERR_INVALID_ARG;
    if (flags & ~(RA_STEP_FIRST | RA_STEP_LAST)) return RA_ERR_INVALID_ARG;
    const bool first = flags & RA_STEP_FIRST, last = flags & RA_STEP_LAST;
    if (empty_problem(B, Sb)) return RA_OK;
    if (!q || !k || !v) return RA_ERR_INVALID_ARG;
    // the state is read unless this is the first fold, written unless the last
    if (!(first && last) && (!state_o || !state_lse)) return RA_ERR_INVALID_ARG;
    if (last && !out) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (state_o && !aligned16(state_o)) ||
        (state_lse && !aligned16(state_lse)) || (out && !aligned16(out)) ||
        (lse && !aligned16(lse)))
        return RA_ERR_ALIGN;
    ra::StepProblem p;
    p.q = q; p.k = k; p.v = v;
    p.state_o = state_o; p.state_lse = state_lse; p.out = out; p.lse = lse;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sb = Sb; p.D = D; p.N = N; p.i = i; p.j = j;
    p.causal = causal ? 1 : 0;
    p.layout = layout;
    p.scale = (scale > 0.f && std::isfinite(scale)) ? scale : (float)(1.0 / std::sqrt((double)D));
    p.first = first ? 1 : 0;
    p.last = last ? 1 : 0;
    if (!ra::tc_step_supported(p)) return RA_ERR_UNSUPPORTED;
    unsigned int* status = nullptr;
    int sms = 0;
    int rc = device_state(&status, &sms);
    if (rc) return rc;
    unsigned int* work = nullptr;
    if ((rc = work_slot(&work))) return rc;
    rc = ra::launch_tc_step(p, status, work, sms, static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_ring_step_backward(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* dout, float* delta, float* dq_state,
                          float* dk_state, float* dv_state, void* dq, void* dk, void* dv, int B,
                          int Hq, int Hkv, int64_t Sb, int D, int N, int i, int j, int causal,
                          int layout, float scale, int flags, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sb < 0 || D <= 0 || N <= 0) return RA_ERR_INVALID_ARG;
    if (Hq % Hkv || i < 0 || i >= N || j < 0 || j >= N) return RA_ERR_INVALID_ARG;
    if (layout < RA_LAYOUT_CONTIGUOUS || layout > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    if (layout == RA_LAYOUT_ZIGZAG && Sb % 2) return RA_ERR_INVALID_ARG;
    if (flags & ~(RA_STEP_FIRST | RA_STEP_LAST)) return RA_ERR_INVALID_ARG;
    const bool first = flags & RA_STEP_FIRST, last = flags & RA_STEP_LAST;
    if (empty_problem(B, Sb)) return RA_OK;
    if (!q || !k || !v || !lse || !dout || !delta) return RA_ERR_INVALID_ARG;
    if (first && !out) return RA_ERR_INVALID_ARG;  // delta comes from out and dout
    // the state is read unless this is the first step, written unless the last
    if (!(first && last) && (!dq_state || !dk_state || !dv_state)) return RA_ERR_INVALID_ARG;
    if (last && (!dq || !dk || !dv)) return RA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, out, lse, dout, delta, dq_state, dk_state, dv_state, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (ptr && !aligned16(ptr)) return RA_ERR_ALIGN;
    ra::BwdStepProblem p;
    p.q = q; p.k = k; p.v = v; p.out = out; p.lse = lse; p.dout = dout; p.delta = delta;
    p.dq_state = dq_state; p.dk_state = dk_state; p.dv_state = dv_state;
    p.dq = dq; p.dk = dk; p.dv = dv;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sb = Sb; p.D = D; p.N = N; p.i = i; p.j = j;
    p.causal = causal ? 1 : 0;
    p.layout = layout;
    p.scale = (scale > 0.f && std::isfinite(scale)) ? scale : (float)(1.0 / std::sqrt((double)D));
    p.first = first ? 1 : 0;
    p.last = last ? 1 : 0;
    if (!ra::tc_bwd_step_supported(p)) return RA_ERR_UNSUPPORTED;
    unsigned int* status = nullptr;
    int sms = 0;
    int rc = device_state(&status, &sms);
    if (rc) return rc;
    unsigned int* work = nullptr;
    if ((rc = work_slot(&work))) return rc;
    rc = ra::launch_bwd_tc_step(p, status, work, sms, static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_watchdog_selftest(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int striped,
                         float scale, int64_t timeout_cycles, void* stream) {
    int rc = validate_forward(q, k, v, out, lse, B, Hq, Hkv, S, D, N, RA_BF16, striped);
    if (rc) return rc;
    if (empty_problem(B, S)) return RA_ERR_INVALID_ARG;  // the self test needs a kernel to run
    if (timeout_cycles < 100000 || timeout_cycles > 4000000000ll) return RA_ERR_INVALID_ARG;
    const ra::FwdProblem p = make_problem(q, k, v, out, lse, B, Hq, Hkv, S, D, N, causal, striped,
                                          scale, RA_BF16);
    if (!ra::tc_supported(p)) return RA_ERR_UNSUPPORTED;
    unsigned int* status = nullptr;
    int sms = 0;
    if ((rc = device_state(&status, &sms))) return rc;
    unsigned int* work = nullptr;
    if ((rc = work_slot(&work))) return rc;
    rc = ra::launch_tc(p, nullptr, status, work, sms, static_cast<cudaStream_t>(stream),
                       timeout_cycles, 1);
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_merge(void* out_a, float* lse_a, const void* out_b, const float* lse_b, int64_t rows,
             int D, int dtype, void* stream) {
    if (rows < 0 || D <= 0 || D > 1024) return RA_ERR_INVALID_ARG;
    if (dtype != RA_BF16 && dtype != RA_F32) return RA_ERR_INVALID_ARG;
    if (rows == 0) return RA_OK;
    if (!out_a || !lse_a || !out_b || !lse_b) return RA_ERR_INVALID_ARG;
    if (!aligned16(out_a) || !aligned16(out_b) || ((uintptr_t)lse_a & 3u) || ((uintptr_t)lse_b & 3u))
        return RA_ERR_ALIGN;
    int rc = device_state(nullptr, nullptr);
    if (rc) return rc;
    rc = ra::launch_merge(out_a, lse_a, out_b, lse_b, rows, D, dtype, static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_relayout(const void* src, void* dst, int64_t BH, int64_t S, int N, int64_t row_bytes,
                int layout, int inverse, void* stream) {
    if (BH < 0 || S < 0 || N <= 0 || row_bytes <= 0 || row_bytes % 4) return RA_ERR_INVALID_ARG;
    if (S % N) return RA_ERR_INVALID_ARG;
    if (layout < RA_LAYOUT_CONTIGUOUS || layout > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    if (layout == RA_LAYOUT_ZIGZAG && (S / N) % 2) return RA_ERR_INVALID_ARG;
    if (BH == 0 || S == 0) return RA_OK;
    if (!src || !dst) return RA_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return RA_ERR_ALIGN;
    const char* s = static_cast<const char*>(src);
    char* d = static_cast<char*>(dst);
    const int64_t bytes = BH * S * row_bytes;
    if (s < d + bytes && d < s + bytes) return RA_ERR_INVALID_ARG;  // overlap
    int rc = device_state(nullptr, nullptr);
    if (rc) return rc;
    rc = ra::launch_stripe(src, dst, BH, S, N, row_bytes, layout, inverse ? 1 : 0,
                           static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_stripe(const void* src, void* dst, int64_t BH, int64_t S, int N, int64_t row_bytes,
              int inverse, void* stream) {
    return ra_relayout(src, dst, BH, S, N, row_bytes, RA_LAYOUT_STRIPED, inverse, stream);
}

int ra_ulysses_exchange(const void* src, void* dst, int B, int H, int64_t S, int N,
                        int64_t row_bytes, int inverse, void* stream) {
    if (B < 0 || H < 0 || S < 0 || N <= 0 || row_bytes <= 0 || row_bytes % 4) return RA_ERR_INVALID_ARG;
    if (S % N || H % N) return RA_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || S == 0) return RA_OK;
    if (!src || !dst) return RA_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return RA_ERR_ALIGN;
    const char* s = static_cast<const char*>(src);
    char* d = static_cast<char*>(dst);
    const int64_t bytes = (int64_t)B * H * S * row_bytes;
    if (s < d + bytes && d < s + bytes) return RA_ERR_INVALID_ARG;  // overlap
    int rc = device_state(nullptr, nullptr);
    if (rc) return rc;
    rc = ra::launch_ulysses(src, dst, B, H, S, N, row_bytes, inverse ? 1 : 0,
                            static_cast<cudaStream_t>(stream));
    if (rc == RA_ERR_CUDA) note_cuda(cudaGetLastError());
    return rc;
}

int ra_plan_tile(int64_t S, int N, int causal, int striped, int tile, int i, int qt,
                 int32_t* items, int64_t cap, int64_t* n_items) {
    if (!n_items || S <= 0 || N <= 0 || tile < 2 || S % N) return RA_ERR_INVALID_ARG;
    if (striped < RA_LAYOUT_CONTIGUOUS || striped > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    const int64_t Sb = S / N;
    // the last tile of a shard may be partial, except under zigzag, whose
    // chunks must be whole tiles
    if (striped == RA_LAYOUT_ZIGZAG && Sb % (2 * tile)) return RA_ERR_INVALID_ARG;
    const int64_t nt = (Sb + tile - 1) / tile;
    if (nt > 0x7fffffff || i < 0 || i >= N || qt < 0 || qt >= nt) return RA_ERR_INVALID_ARG;
    ra::RingGeom g{N, (int)nt, causal ? 1 : 0, striped};
    int64_t n = 0;
    for (int s = 0; s < N; ++s) {
        const int j = ((i - s) % N + N) % N;
        int nk = 0, dk = 0;
        ra::shard_span(g, i, j, qt, &nk, &dk);
        for (int kt = 0; kt < nk; ++kt) {
            if (items && n < cap) {
                int32_t* e = items + n * 4;
                e[0] = s;
                e[1] = j;
                e[2] = kt;
                e[3] = ra::fold_kind(g, i, j, qt, kt);
            }
            ++n;
        }
    }
    *n_items = n;
    return (items && n > cap) ? RA_ERR_CAPACITY : RA_OK;
}

int ra_plan(int64_t S, int N, int causal, int striped, int tile, int32_t* items, int64_t cap,
            int64_t* n_items) {
    if (!n_items || S <= 0 || N <= 0 || tile < 2 || S % N) return RA_ERR_INVALID_ARG;
    if (striped < RA_LAYOUT_CONTIGUOUS || striped > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    const int64_t Sb = S / N;
    if (striped == RA_LAYOUT_ZIGZAG && Sb % (2 * tile)) return RA_ERR_INVALID_ARG;
    const int64_t nt = (Sb + tile - 1) / tile;
    if (nt > 0x7fffffff) return RA_ERR_INVALID_ARG;
    ra::RingGeom g{N, (int)nt, causal ? 1 : 0, striped};
    int64_t n = 0;
    for (int i = 0; i < N; ++i)
        for (int qt = 0; qt < (int)nt; ++qt)
            for (int s = 0; s < N; ++s) {
                const int j = ((i - s) % N + N) % N;
                int nk = 0, dk = 0;
                ra::shard_span(g, i, j, qt, &nk, &dk);
                for (int kt = 0; kt < nk; ++kt) {
                    if (items && n < cap) {
                        int32_t* e = items + n * 6;
                        e[0] = i;
                        e[1] = qt;
                        e[2] = s;
                        e[3] = j;
                        e[4] = kt;
                        e[5] = ra::fold_kind(g, i, j, qt, kt);
                    }
                    ++n;
                }
            }
    *n_items = n;
    return (items && n > cap) ? RA_ERR_CAPACITY : RA_OK;
}

int ra_plan_backward(int64_t S, int N, int causal, int striped, int tile, int j, int kt,
                     int32_t* items, int64_t cap, int64_t* n_items) {
    if (!n_items || S <= 0 || N <= 0 || tile < 2 || S % N) return RA_ERR_INVALID_ARG;
    if (striped < RA_LAYOUT_CONTIGUOUS || striped > RA_LAYOUT_ZIGZAG) return RA_ERR_INVALID_ARG;
    const int64_t Sb = S / N;
    if (striped == RA_LAYOUT_ZIGZAG && Sb % (2 * tile)) return RA_ERR_INVALID_ARG;
    const int64_t nt = (Sb + tile - 1) / tile;
    if (nt > 0x7fffffff || j < 0 || j >= N || kt < 0 || kt >= nt) return RA_ERR_INVALID_ARG;
    ra::RingGeom g{N, (int)nt, causal ? 1 : 0, striped};
    int64_t n = 0;
    ra::KeyWalk w;
    for (w.start(g, j, kt, 1); !w.done(g); w.next(g, j, kt, 1)) {
        if (items && n < cap) {
            int32_t* e = items + n * 4;
            e[0] = w.s;
            e[1] = w.i;
            e[2] = w.qt;
            e[3] = ra::fold_kind(g, w.i, j, w.qt, kt);
        }
        ++n;
    }
    *n_items = n;
    return (items && n > cap) ? RA_ERR_CAPACITY : RA_OK;
}

int ra_check(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) { note_cuda(e); return RA_ERR_CUDA; }
    unsigned int* status = nullptr;
    int rc = device_state(&status, nullptr);
    if (rc) return rc;
    unsigned int st = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&st, g_ra_status, sizeof(st))) != cudaSuccess ||
        (e = cudaMemcpyToSymbol(g_ra_status, &zero, sizeof(zero))) != cudaSuccess) {
        note_cuda(e);
        return RA_ERR_CUDA;
    }
    if (st & ra::kStatusTimeout) return RA_ERR_TIMEOUT;
    if (st & ra::kStatusBounds) return RA_ERR_BOUNDS;
    return RA_OK;
}

const char* ra_strerror(int code) {
    switch (code) {
        case RA_OK: return "ok";
        case RA_ERR_INVALID_ARG: return "invalid argument";
        case RA_ERR_UNSUPPORTED: return "unsupported shape, dtype or device";
        case RA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case RA_ERR_CUDA: return g_cuda_msg[0] ? g_cuda_msg : "CUDA runtime error";
        case RA_ERR_TIMEOUT: return "a kernel wait timed out";
        case RA_ERR_BOUNDS: return "a kernel bounds check failed";
        case RA_ERR_CAPACITY: return "output array too small";
        default: return "unknown status";
    }
}

int ra_tile_config(int* tq, int* tk) {
    if (tq) *tq = 128;
    if (tk) *tk = 128;
    return RA_OK;
}

int ra_version(void) { return 100; }

}  // extern "C"
