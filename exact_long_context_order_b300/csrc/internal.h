// Internal launch interface between the C-ABI layer (ra_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace ra {

// Bits of the device status word (one per device, read by ra_check).
enum : unsigned int { kStatusTimeout = 1u, kStatusBounds = 2u };

struct FwdProblem {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    float* lse;
    int B, Hq, Hkv;
    int64_t S;
    int D, N, causal, striped;  // striped: layout 0 contiguous, 1 striped, 2 zigzag
    float scale;  // resolved (> 0)
    int dtype;    // RA_BF16 / RA_F32
};

struct FoldLog {
    int32_t* log;
    int32_t* counts;
    int max_entries;
};

// Returns 0 on success or an RA_ERR_* code.  status: device pointer to this
// device's status word.  sm_count: multiprocessors of the current device.
// work: device counter the kernel takes work items from; zeroed by launch_tc
// on `stream` before the launch.  timeout_cycles (<= 0: the default of 4e9
// SM cycles) bounds every wait of the kernel; withhold_first_k = 1 is the
// failure-detection self test (each CTA's first K-tile copy is never issued,
// so its waits run out and the kernel reports kStatusTimeout).
// split_mode 1 lets a non-causal problem with one to two items per SM run
// as stream-K (fixed contiguous work ranges per CTA; an item cut between two
// CTAs is combined from the tail's partial, scratch taken from a library
// memory pool on `stream`); 0 always uses the dynamic queue.
int launch_tc(const FwdProblem& p, const FoldLog* flog, unsigned int* status, unsigned int* work,
              int sm_count, cudaStream_t stream, long long timeout_cycles = 0,
              int withhold_first_k = 0, int split_mode = 0);
// Whether launch_tc with split_mode 1 runs p as stream-K (host only).
bool tc_uses_streamk(const FwdProblem& p, int sm_count);
bool tc_supported(const FwdProblem& p);
// Device address of the current device's status word (read by ra_check).
int device_status_word(unsigned int** status);
// The current device's status word address and SM count, resolved once per
// device (RA_ERR_UNSUPPORTED unless the device is sm_103).
int device_info(unsigned int** status, int* sm_count);
// Keeps the text of a CUDA error for ra_strerror(RA_ERR_CUDA) (per thread).
void note_cuda_error(cudaError_t e);
int launch_simt(const FwdProblem& p, unsigned int* status, cudaStream_t stream);
// Host-only envelope checks, made before any CUDA call.
bool simt_supported(const FwdProblem& p);
int launch_merge(void* out_a, float* lse_a, const void* out_b, const float* lse_b, int64_t rows,
                 int D, int dtype, cudaStream_t stream);
// layout: 1 striped, 2 zigzag (0 contiguous is the identity)
int launch_stripe(const void* src, void* dst, int64_t BH, int64_t S, int N, int64_t row_bytes,
                  int layout, int inverse, cudaStream_t stream);

// One step of a ring whose devices are separate processes: query shard i
// ([B, Hq, Sb, D]) folds key/value block j ([B, Hkv, Sb, D]) of a ring of N
// devices into its running state (state_o fp32 [B, Hq, Sb, D], state_lse
// [B, Hq, Sb]); on the last step the folded result goes to out (bf16) and lse
// instead of the state.
struct StepProblem {
    const void* q;
    const void* k;
    const void* v;
    float* state_o;
    float* state_lse;
    void* out;
    float* lse;
    int B, Hq, Hkv;
    int64_t Sb;
    int D, N, i, j, causal, layout;
    float scale;  // resolved (> 0)
    int first, last;
};
bool tc_step_supported(const StepProblem& p);
int launch_tc_step(const StepProblem& p, unsigned int* status, unsigned int* work, int sm_count,
                   cudaStream_t stream);

// Backward problem: the forward's tensors plus dout, the gradients and the
// per-row terms delta (float32 [B*Hq*S], in the caller's workspace).
struct BwdProblem {
    const void* q;
    const void* k;
    const void* v;
    const void* out;
    const float* lse;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    float* delta;
    int B, Hq, Hkv;
    int64_t S;
    int D, N, causal, striped;
    float scale;
    int dtype;
};

// One backward step of a ring whose devices are separate processes: query
// shard i (q, out, dout, lse, delta) against the block j it holds (k, v);
// dq_state for the shard, dk_state / dv_state for the block (fp32
// accumulators); on the last step the totals go to dq, dk, dv (bf16).
struct BwdStepProblem {
    const void* q;
    const void* k;
    const void* v;
    const void* out;
    const float* lse;
    const void* dout;
    float* delta;
    float* dq_state;
    float* dk_state;
    float* dv_state;
    void* dq;
    void* dk;
    void* dv;
    int B, Hq, Hkv;
    int64_t Sb;
    int D, N, i, j, causal, layout;
    float scale;  // resolved (> 0)
    int first, last;
};
bool tc_bwd_step_supported(const BwdStepProblem& p);
int launch_bwd_tc_step(const BwdStepProblem& p, unsigned int* status, unsigned int* work,
                       int sm_count, cudaStream_t stream);

int launch_bwd_delta(const BwdProblem& p, cudaStream_t stream);
int launch_bwd_simt(const BwdProblem& p, cudaStream_t stream);
int launch_bwd_dkdv_simt(const BwdProblem& p, cudaStream_t stream);
bool tc_bwd_supported(const BwdProblem& p);
bool simt_bwd_supported(const BwdProblem& p);
bool bwd_delta_supported(const BwdProblem& p);
// Tensor-core backward (delta already computed): the dq kernel, then the
// dk/dv kernel, each zeroing the work counter on `stream` before it starts.
int launch_bwd_tc(const BwdProblem& p, unsigned int* status, unsigned int* work, int sm_count,
                  cudaStream_t stream);
// Failure-detection self test of one backward kernel (which: 0 dq, 1 dk/dv):
// its first K (dq) or Q (dk/dv) tile is never loaded and every wait is
// bounded by timeout_cycles, so the kernel reports kStatusTimeout and returns.
int launch_bwd_tc_selftest(const BwdProblem& p, unsigned int* status, unsigned int* work,
                           int sm_count, cudaStream_t stream, long long timeout_cycles, int which);

int launch_ulysses(const void* src, void* dst, int64_t B, int64_t H, int64_t S, int N,
                   int64_t row_bytes, int inverse, cudaStream_t stream);

}  // namespace ra
