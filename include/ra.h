/*
 * ra.h -- C ABI of the ring-attention library (libra.so), sm_103a.
 *
 * The library computes exact blockwise ring attention on one GPU.  The
 * sequence of S tokens is held by N virtual ring devices (shards) that live
 * side by side in device memory; query shard i visits the key/value shards
 * in ring order j = (i - s) mod N, s = 0..N-1, and folds every block into an
 * online-softmax state (running max, running normaliser, rescaled
 * numerator), so the result equals full softmax attention.
 *   Method: "Ring Attention" glossary page (ultralytics.com), section "Como
 *   funciona a atencao em anel" (ring schedule j = (i - step) mod N,
 *   accumulated exponentiated scores and weighted values, divided at the
 *   end; running-max subtraction in production kernels; causal masking and
 *   Striped Attention); "Sequence parallelism and ring attention"
 *   (aiunderstanding.org), sections "Immersione profonda" (contiguous token
 *   blocks, K/V passed around the ring) and "Approfondimento tecnico"
 *   (online softmax, exact result); "Ring Attention la gi?" (thienlv.com),
 *   section "Uu Diem" (GQA compatibility).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor arguments are DEVICE pointers to memory the caller owns; the
 *   library never frees or keeps them.  Besides one status word per device
 *   (a static __device__ variable created with the module), the library
 *   allocates one 4 KiB block per device on the first tensor-core launch on
 *   that device (cudaMalloc, kept until exit): 64 work-queue counters, one
 *   per launch in flight, each zeroed on the launch's stream.  Make the first
 *   such call on a device outside CUDA-graph stream capture.  A forward run
 *   as stream-K (see ra_forward_ex) also takes scratch, on its stream, from a
 *   memory pool the library creates per device on first use.
 * - Layout is "shard-major": q and out are [B, Hq, S, D], k and v are
 *   [B, Hkv, S, D], lse is [B, Hq, S]; all row-major and contiguous.  Shard i
 *   owns rows [i*Sb, (i+1)*Sb) of every (b, h) slice, Sb = S / N.  The
 *   argument `striped` selects which tokens a shard holds (RA_LAYOUT_*):
 *     0 contiguous: row p holds token p;
 *     1 striped:    row r of shard i holds token r*N + i (token t on shard
 *                   t mod N; the glossary page's Striped Attention);
 *     2 zigzag:     the sequence is cut into 2N chunks of Sb/2 tokens and
 *                   shard i holds chunk i followed by chunk 2N-1-i (a
 *                   variant the Zulu aiunderstanding.org page only names;
 *                   this is the library's reading).  Needs Sb even.
 *   ra_relayout (ra_stripe for the striped layout) converts between token
 *   order and a shard-major layout.
 * - Query head h reads key/value head h / (Hq / Hkv) (grouped-query
 *   attention; Hq must be a multiple of Hkv).
 * - causal = 1 masks every key whose token position is after the query's
 *   (inclusive causal: a query sees its own key).
 * - scale <= 0 selects 1/sqrt(D).
 * - dtype: RA_BF16 (inputs/outputs bfloat16, fp32 accumulation) or RA_F32
 *   (inputs/outputs float32, fp32 arithmetic, no TF32).
 * - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call that takes a stream is asynchronous on it: it validates its
 *   arguments on the host, enqueues kernels and returns.  Device-side
 *   failures (a bounded wait that ran out, a bounds check) are recorded in the
 *   device status word and reported by ra_check.
 * - Return value: RA_OK or one of the error codes below.  On an error
 *   detected on the host nothing is enqueued and no output is touched.
 */
#ifndef RA_H_
#define RA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, S % N, Hq % Hkv, ... */
    RA_ERR_UNSUPPORTED = 2, /* shape/dtype/device the kernels do not handle */
    RA_ERR_ALIGN = 3,       /* pointer not 16-byte aligned */
    RA_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, ...) */
    RA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (reported by ra_check) */
    RA_ERR_BOUNDS = 6,      /* a kernel's bounds check failed (reported by ra_check) */
    RA_ERR_CAPACITY = 7     /* a caller-provided output array is too small */
};

enum { RA_BF16 = 0, RA_F32 = 1 };

enum { RA_LAYOUT_CONTIGUOUS = 0, RA_LAYOUT_STRIPED = 1, RA_LAYOUT_ZIGZAG = 2 };

/* Kernel selection for ra_forward_ex. */
enum {
    RA_KERNEL_AUTO = 0, /* tensor-core kernel when the shape allows it, else SIMT */
    RA_KERNEL_TC = 1,   /* tcgen05 tensor-core kernel (bf16, D in {64,128}; any Sb for
                           contiguous/striped shards, Sb % 256 == 0 for zigzag) */
    RA_KERNEL_SIMT = 2  /* fp32 SIMT kernel (any D <= 256, any Sb); f32 or bf16 */
};

/* Flags of ra_ring_step. */
enum { RA_STEP_FIRST = 1, RA_STEP_LAST = 2 };

/* Fold kinds reported by ra_plan / ra_fold_log. */
enum { RA_FOLD_FULL = 0, RA_FOLD_INCL = 1, RA_FOLD_STRICT = 2 };

/*
 * ra_forward: out = softmax(scale * Q K^T [masked]) V over the ring.
 *   q   [B, Hq, S, D]  (read)      k, v [B, Hkv, S, D]  (read)
 *   out [B, Hq, S, D]  (written)   lse  [B, Hq, S] float32, natural log of the
 *                                  softmax normaliser per query row
 *                                  (written; may be NULL)
 *   Hq, Hkv, D, N > 0; B, S >= 0; S % N == 0; Hq % Hkv == 0.  An empty
 *   problem (B == 0 or S == 0) is a no-op that returns RA_OK without any
 *   CUDA call; its buffer pointers may then be NULL.
 * Computes, for each query shard i, the fold over ring steps s = 0..N-1 of
 * key/value shard j = (i - s) mod N (glossary page, "Como funciona": the
 * schedule and the numerator/denominator fold; aiunderstanding.org,
 * "Approfondimento tecnico": running max and normaliser with rescaling).
 * Under causal masking whole shards and key tiles with no visible pair are
 * skipped, never computed.  When the key/value shards that the query shards
 * in flight at once would read together exceed the L2 (striped, zigzag and
 * non-causal layouts at very long S, e.g. 1M tokens in 64 shards), the
 * tensor-core kernel enters every query shard's ring at shard N-1: query
 * shard i then folds j = N-1, N-2, ..., 0, the same cyclic order from ring
 * step (i + 1) mod N, so that all of them read one key/value shard at a
 * time.  Only the rounding of the fold can differ.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_ALIGN (q, k, v, out, lse not 16-byte
 * aligned), RA_ERR_UNSUPPORTED (D > 256, device not sm_103, or a shape that
 * no kernel takes: the tensor-core kernel needs B*Hq*S and B*Hkv*S below 2^31
 * rows, the SIMT kernel B*Hq and N at most 65535; decided on the host before
 * any CUDA call), RA_ERR_CUDA.
 */
int ra_forward(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
               int Hkv, int64_t S, int D, int N, int causal, int striped, float scale, int dtype,
               void* stream);

/*
 * ra_forward_host: ra_forward on host tensors.  Enqueues the copies of q, k,
 * v from host to the caller's device staging buffers, the forward, and the
 * copies of out (and lse, when lse_host is not NULL) back to the host.
 * With at least four (batch, KV head) groups (B*Hkv >= 4) the call pipelines
 * up to eight chunks of consecutive groups: chunk c+1's copies in overlap
 * chunk c's forward, and chunk c's copies out overlap later chunks'.  (A
 * chunk starts at an offset of whole groups into each staging buffer; if one
 * such offset is not a multiple of 16 bytes, or ra_forward would run the
 * problem as stream-K (see ra_forward_ex), the call runs in order instead.)
 * That
 * work runs on streams the library creates for the device on first use (one
 * copy stream per direction, two compute streams, kept until the process
 * exits), forked from `stream` at the start of the call and joined back into
 * it at the end, so `stream` orders the whole call as if it ran there (also
 * when an error stops the call part-way: what was enqueued is joined before
 * the error is returned); the outputs are the bits ra_forward computes.  Concurrent calls from several
 * host threads are serialised while they enqueue.  Fewer groups run in order
 * on `stream` itself.  Asynchronous: the host buffers must stay valid until
 * `stream` reaches the end of the call; page-locked (pinned) host memory
 * makes the copies asynchronous.
 *   q_host, k_host, v_host (read), out_host, lse_host (written; lse_host may
 *   be NULL, then lse_dev must be NULL too): host memory with the layouts of
 *   ra_forward.
 *   q_dev, k_dev, v_dev, out_dev, lse_dev: device staging buffers of the same
 *   sizes (caller-owned, 16-byte aligned), overwritten.
 * Errors: as ra_forward; RA_ERR_INVALID_ARG for a NULL host pointer (of a
 * non-empty problem) or an lse pair with one NULL; RA_ERR_CUDA when a copy
 * cannot be enqueued.
 */
int ra_forward_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                    float* lse_host, void* q_dev, void* k_dev, void* v_dev, void* out_dev,
                    float* lse_dev, int B, int Hq, int Hkv, int64_t S, int D, int N, int causal,
                    int striped, float scale, int dtype, void* stream);

/* ra_forward with an explicit kernel choice (RA_KERNEL_*).  RA_KERNEL_TC
 * returns RA_ERR_UNSUPPORTED when the shape is outside its envelope.
 * Stream-K.  The tensor-core kernel runs one persistent CTA per SM and hands
 * out work items (pairs of 128-row query tiles, each folding its whole ring)
 * from a queue.  A non-causal problem with between one and two items per SM
 * would leave many SMs idle in the queue's last wave, so RA_KERNEL_AUTO then
 * gives every CTA an equal, contiguous range of the items' key tiles
 * instead.  An item cut between two CTAs is folded as a head and a tail
 * segment; the tail writes its partial (O/l and lse, fp32) and the head,
 * which finishes later, combines it with its own by the log-sum-exp
 * weighting of ra_merge -- the same two halves in the same order on every
 * call, so the result does not depend on timing.  The scratch (2*128 rows of
 * D + 1 floats per item) is taken on `stream` from a memory pool the library
 * owns per device (created on first use; freed blocks stay reserved, up to
 * 1 GiB, for reuse); under CUDA-graph stream capture it is a graph
 * allocation.  RA_KERNEL_TC always uses the queue.  A head waits only for
 * its successor CTA's first segment, and CTAs start in index order, so the
 * kernel completes even when it shares the GPU with other work; the wait is
 * bounded (4e9 SM cycles, about 2 s) and could run out only if other kernels
 * kept the successor off every SM for that long: ra_check then reports
 * RA_ERR_TIMEOUT. */
int ra_forward_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                  int Hq, int Hkv, int64_t S, int D, int N, int causal, int striped, float scale,
                  int dtype, int kernel, void* stream);

/*
 * ra_ring_step: one step of a ring whose devices are separate processes (or
 * GPUs): query shard i folds the key/value block j it holds at this step into
 * its running online-softmax state.  This is the per-device step of the
 * method: device i keeps its query block, at ring step s it holds block
 * j = (i - s) mod N received from the previous device, computes the scores
 * of its queries against that block and folds them into a running maximum,
 * normaliser and rescaled numerator (glossary page, "Como funciona a atencao
 * em anel"; aiunderstanding.org, "Immersione profonda": only K and V travel
 * round the ring, the transfer hidden behind the block's compute, and
 * "Approfondimento tecnico": the online-softmax fold).  Moving the block
 * between devices is the caller's (the package's ring driver uses
 * torch.distributed send/recv); this call only computes.
 *   q        [B, Hq, Sb, D] bf16 (read): query shard i.
 *   k, v     [B, Hkv, Sb, D] bf16 (read): key/value block j.
 *   state_o  [B, Hq, Sb, D] float32, state_lse [B, Hq, Sb] float32: the
 *            running state, the normalised output and natural-log
 *            log-sum-exp of the blocks folded so far (-inf, output 0, for a
 *            row that has seen no visible key).  Read unless RA_STEP_FIRST,
 *            written unless RA_STEP_LAST; may be NULL when both flags are set.
 *   out      [B, Hq, Sb, D] bf16, lse [B, Hq, Sb] float32: written only with
 *            RA_STEP_LAST (the state after this fold, as ra_forward's outputs
 *            for shard i); out must then be given, lse may be NULL.
 *   Sb: tokens per shard (any Sb >= 0 for contiguous and striped shards;
 *   zigzag needs Sb % 256 == 0).  N: ring devices; 0 <= i, j < N.  causal,
 *   layout (RA_LAYOUT_*), scale: as ra_forward, applied to the global token
 *   positions of shard i's queries and block j's keys, so folding blocks
 *   j = i, i-1, ..., i-N+1 (mod N) with the first flagged RA_STEP_FIRST and
 *   the last RA_STEP_LAST gives ra_forward's result for shard i.  A block
 *   with no visible pair leaves the state as it was.
 *   flags: RA_STEP_FIRST | RA_STEP_LAST (both for N = 1).
 * The fold of a block's partial (O_b, lse_b) into the state (O_s, lse_s) is
 * the log-sum-exp weighting of ra_merge, in fp32:
 *   lse = ln(e^lse_s + e^lse_b),  O = e^(lse_s-lse) O_s + e^(lse_b-lse) O_b.
 * Runs the tcgen05 tensor-core kernel (bf16, D in {64, 128}).
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_ALIGN (any pointer not 16-byte
 * aligned), RA_ERR_UNSUPPORTED (D, device, or B*Hq*Sb >= 2^31 rows),
 * RA_ERR_CUDA.  An empty problem (B == 0 or Sb == 0) is a no-op.
 */
int ra_ring_step(const void* q, const void* k, const void* v, float* state_o, float* state_lse,
                 void* out, float* lse, int B, int Hq, int Hkv, int64_t Sb, int D, int N, int i,
                 int j, int causal, int layout, float scale, int flags, void* stream);

/*
 * ra_ring_step_backward: one step of the backward of a ring whose devices are
 * separate processes (or GPUs), the counterpart of ra_ring_step for
 * training.  Device i keeps its query shard and, at ring step s, holds block
 * j = (i - s) mod N together with that block's gradient accumulators, which
 * travel with it (the glossary page's ring, "Como funciona a atencao em
 * anel"; the backward is the chain rule of ra_backward's definition, folded
 * block by block): this call adds block j's terms into the shard's dq and
 * the shard's terms into the block's dk and dv.
 *   q, out, dout [B, Hq, Sb, D] bf16 (read): shard i's queries, the
 *       forward's output and dL/dout for them.  out is read on the first step
 *       only.
 *   lse [B, Hq, Sb] float32 (read): the forward's lse for the shard.
 *   delta [B, Hq, Sb] float32 (caller-owned): written on the first step
 *       (rowsum(dout * out)), read by every step.
 *   k, v [B, Hkv, Sb, D] bf16 (read): block j.
 *   dq_state [B, Hq, Sb, D] float32: the shard's running dq (scaled);
 *   dk_state, dv_state [B, Hkv, Sb, D] float32: block j's running dk
 *       (scaled) and dv, which the caller passes on with the block.  Read
 *       unless flags has RA_STEP_FIRST (then they start at zero), written
 *       unless flags has RA_STEP_LAST; may be NULL when both flags are set.
 *   dq, dk, dv (bf16, written on the last step only, may be NULL otherwise):
 *       the totals of the shard's dq and of block j's dk and dv; the block's
 *       then travel one more hop, to the device that holds block j.
 *   i, j, N, causal, layout, scale: as ra_ring_step.  Every device calls
 *       with RA_STEP_FIRST at s = 0 and RA_STEP_LAST at s = N - 1.
 * Masks, tiles and kernels are those of ra_backward's tensor-core kernels
 * (bf16, D in {64, 128}; Sb % 256 == 0 for zigzag), compiled for one block:
 * the dq kernel over the shard's query tiles, the dk/dv kernel over the
 * block's key tiles.  A tile pair no query of the shard sees leaves the
 * state as it was.  Asynchronous on `stream`; no atomics (the same bits on
 * every call).
 * Errors: RA_ERR_INVALID_ARG (shapes, i or j out of range, flags, a NULL
 * pointer the flags need), RA_ERR_ALIGN, RA_ERR_UNSUPPORTED, RA_ERR_CUDA.  An
 * empty problem (B == 0 or Sb == 0) is a no-op.
 */
int ra_ring_step_backward(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* dout, float* delta, float* dq_state,
                          float* dk_state, float* dv_state, void* dq, void* dk, void* dv, int B,
                          int Hq, int Hkv, int64_t Sb, int D, int N, int i, int j, int causal,
                          int layout, float scale, int flags, void* stream);

/*
 * ra_merge: fold partial result b into partial result a, in place.
 *   out_a [rows, D] (read, written)   lse_a [rows] float32 (read, written)
 *   out_b [rows, D] (read)            lse_b [rows] float32 (read)
 * Each partial is a normalised attention output over a disjoint key set
 * with its log-sum-exp; the result is the attention over the union:
 *   lse = ln(e^lse_a + e^lse_b),  out_a = e^(lse_a-lse) out_a + e^(lse_b-lse) out_b
 * (the same rescale-and-add the online softmax performs when a block arrives;
 * aiunderstanding.org, "Approfondimento tecnico").  A partial with
 * lse = -inf contributes nothing; two empty partials give out 0, lse -inf.
 * dtype RA_BF16 or RA_F32 for out_a/out_b.  rows >= 0, 0 < D <= 1024.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_ALIGN, RA_ERR_CUDA.
 */
int ra_merge(void* out_a, float* lse_a, const void* out_b, const float* lse_b, int64_t rows,
             int D, int dtype, void* stream);

/*
 * ra_stripe: permute rows between token order and striped shard-major order.
 *   src, dst: [BH, S, row_bytes] byte arrays (device; must not overlap).
 *   inverse = 0: dst[i*Sb + r] = src[r*N + i]   (token order -> striped shards)
 *   inverse = 1: dst[r*N + i] = src[i*Sb + r]   (striped shards -> token order)
 * for every (bh) slice; Sb = S / N (glossary page, Striped Attention: tokens
 * spread evenly over the devices, read as token t -> shard t mod N).
 * row_bytes > 0 and a multiple of 4.  Bit-exact copy.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_ALIGN (pointers not 16-byte aligned),
 * RA_ERR_CUDA.
 */
int ra_stripe(const void* src, void* dst, int64_t BH, int64_t S, int N, int64_t row_bytes,
              int inverse, void* stream);

/*
 * ra_relayout: permute rows between token order and a shard-major layout.
 *   src, dst: [BH, S, row_bytes] byte arrays (device; must not overlap).
 *   layout: RA_LAYOUT_* (contiguous is a plain copy).
 *   inverse = 0: dst row p = src row (token held by shard-major row p)
 *                (token order -> shard-major)
 *   inverse = 1: dst row t = src row (shard-major row holding token t)
 *                (shard-major -> token order)
 * for every (bh) slice.  row_bytes > 0 and a multiple of 4.  Bit-exact copy.
 * Errors: RA_ERR_INVALID_ARG (also: unknown layout, zigzag with odd S/N),
 * RA_ERR_ALIGN (pointers not 16-byte aligned), RA_ERR_CUDA.
 */
int ra_relayout(const void* src, void* dst, int64_t BH, int64_t S, int N, int64_t row_bytes,
                int layout, int inverse, void* stream);

/*
 * ra_ulysses_exchange: the head/sequence all-to-all of DeepSpeed Ulysses,
 * the alternative context-parallel scheme the glossary page contrasts with
 * ring attention ("Atencao em anel vs. outros tipos de paralelismo": every
 * device receives all tokens of a subset of the heads), as a permutation
 * between N device-contiguous buffers on one GPU.
 *   inverse = 0: src sequence-sharded [N][B][H][S/N][row_bytes] (device i
 *                holds tokens [i*S/N, (i+1)*S/N) of every head) ->
 *                dst head-sharded [N][B][H/N][S][row_bytes] (device d holds
 *                heads [d*H/N, (d+1)*H/N), all tokens in order):
 *                dst[d][b][hl][t] = src[t/(S/N)][b][d*H/N + hl][t%(S/N)]
 *   inverse = 1: the reverse permutation.
 * Device d's head-sharded buffer is an ra_forward input ([B, H/N, S, D],
 * contiguous layout, one ring device), so exchange -> attention -> inverse
 * exchange is Ulysses attention.  Requires S % N == 0 and H % N == 0;
 * row_bytes > 0 and a multiple of 4; src and dst must not overlap.
 * Bit-exact copy.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_ALIGN, RA_ERR_CUDA, RA_ERR_UNSUPPORTED
 * (more than 65535 chunks, B*H*N).
 */
int ra_ulysses_exchange(const void* src, void* dst, int B, int H, int64_t S, int N,
                        int64_t row_bytes, int inverse, void* stream);

/*
 * ra_plan (host only, no GPU): the whole fold schedule of the ring, the
 * ordered work list the kernels follow.  Writes n_items entries of 6 int32
 * each, (i, qt, s, j, kt, kind): query shards i ascending, their query tiles
 * qt ascending (rows [qt*tile, (qt+1)*tile) of the shard), and for each query
 * tile its folds in order -- ring steps s ascending with j = (i - s) mod N
 * (glossary page, "Como funciona a atencao em anel": device i holds block
 * (i - step) mod N, received from the previous device), key tiles kt of
 * shard j ascending -- listing only tiles that hold at least one visible
 * (query, key) pair, so the causal block and tile skips are the entries
 * that are absent.  kind is RA_FOLD_FULL (every pair visible), RA_FOLD_INCL
 * (pairs with local key row <= local query row) or RA_FOLD_STRICT (local
 * key row < local query row).  The tensor-core kernel folds every query
 * tile in exactly this order (ra_fold_log records it), or in ra_forward's
 * long-sequence case in this order rotated to start at ring step
 * (i + 1) mod N (see ra_forward).
 *   items: int32[cap][6] or NULL (then only *n_items is set).
 *   striped is the layout (RA_LAYOUT_*).  Requires tile >= 2; a shard's last
 *   tile may be partial (ceil(Sb/tile) tiles), except under zigzag, which
 *   needs Sb % (2*tile) == 0.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_CAPACITY (cap too small; *n_items is
 * still set).
 */
int ra_plan(int64_t S, int N, int causal, int striped, int tile, int32_t* items, int64_t cap,
            int64_t* n_items);

/*
 * ra_plan_tile (host only, no GPU): the fold list of one query tile, the
 * entries of ra_plan whose (i, qt) are given.  For query shard i and query
 * tile qt writes n_items entries of 4 int32 each, (s, j, kt, kind), in fold
 * order.
 *   items: int32[cap][4] or NULL (then only *n_items is set).  Same size
 *   rules as ra_plan; 0 <= i < N, 0 <= qt < ceil(Sb/tile).
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_CAPACITY (cap too small; *n_items is
 * still set).
 */
int ra_plan_tile(int64_t S, int N, int causal, int striped, int tile, int i, int qt,
                 int32_t* items, int64_t cap, int64_t* n_items);

/*
 * ra_plan_backward (host only, no GPU): the visiting order of one key tile in
 * the backward's dk/dv pass.  For key tile kt of shard j (rows
 * [kt*tile, (kt+1)*tile) of the shard), writes n_items entries of 4 int32,
 * (s, i, qt, kind).  The block and the gradient accumulators travelling with
 * it go round the ring in its cyclic order, entering it at device 0: query
 * shards i = 0, 1, ..., N-1 ascending, s = (i - j) mod N being the ring step
 * at which block j reaches device i; then the query tiles qt of shard i that
 * hold at least one (query, key) pair the mask leaves visible, ascending;
 * kind as in ra_plan for the pair (query tile qt of shard i, key tile kt of
 * shard j).
 * Every query head of the GQA group is visited with the same list (heads
 * between the step and the query tiles).  Each pair appears exactly once
 * across the key tiles, as in ra_plan.
 *   items: int32[cap][4] or NULL.  Same size rules as ra_plan.
 * Errors: RA_ERR_INVALID_ARG, RA_ERR_CAPACITY (*n_items is still set).
 */
int ra_plan_backward(int64_t S, int N, int causal, int striped, int tile, int j, int kt,
                     int32_t* items, int64_t cap, int64_t* n_items);

/*
 * ra_fold_log: run the tensor-core kernel in its logging variant and record
 * the order in which each query tile was folded.
 *   Same tensor arguments as ra_forward (bf16 only).
 *   log: device int32 buffer of B*Hq*N*nt * max_entries * 4 entries, with
 *        nt = ceil(Sb/128) query tiles per shard.  For the query tile
 *        (b, h, i, qt), at index ((b*Hq + h)*N + i)*nt + qt, entry n is
 *        (s, j, kt, kind) of its n-th live fold; unused entries are left as
 *        written by the caller.
 *   counts: device int32[B*Hq*N*nt]: number of live folds recorded per tile.
 *   max_entries >= N * nt.
 * The logging variant always folds in ring order, so it computes the same
 * outputs as ra_forward except where ra_forward enters the ring at shard
 * N-1 (there they agree up to rounding).
 * Errors: as ra_forward, plus RA_ERR_UNSUPPORTED outside the tensor-core
 * kernel's envelope and RA_ERR_INVALID_ARG for an empty problem.
 */
int ra_fold_log(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
                int Hkv, int64_t S, int D, int N, int causal, int striped, float scale,
                int32_t* log, int32_t* counts, int max_entries, void* stream);

/*
 * ra_watchdog_selftest: failure-detection self test of the tensor-core
 * kernel.  It launches the kernel on the caller's problem (same arguments as
 * ra_forward, bf16, tensor-core shapes) with every wait bounded by
 * timeout_cycles SM clock cycles (1e5 .. 4e9) and with each CTA's first K-tile
 * copy never issued, so the waits that depend on it run out.  The kernel then
 * records RA_ERR_TIMEOUT in the device status word, lets its copies and MMAs
 * in flight finish, frees its tensor memory and returns; nothing faults or
 * hangs and the CUDA context stays usable.  out and lse are left undefined.
 * Returns RA_OK once the launch is enqueued; ra_check(stream) then reports
 * RA_ERR_TIMEOUT.  (Normal launches bound every wait at 4e9 cycles.)
 * Errors: as ra_forward; RA_ERR_INVALID_ARG for timeout_cycles out of range
 * or an empty problem (the test needs a kernel to run).
 */
int ra_watchdog_selftest(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int striped,
                         float scale, int64_t timeout_cycles, void* stream);

/*
 * ra_backward: gradients of ra_forward with respect to q, k and v.
 *   q, k, v [shapes of ra_forward] (read): the forward's inputs.
 *   out [B, Hq, S, D] (read), lse [B, Hq, S] float32 (read, not NULL): the
 *       forward's outputs for these inputs.
 *   dout [B, Hq, S, D] (read): dL/dout.
 *   dq [B, Hq, S, D], dk [B, Hkv, S, D], dv [B, Hkv, S, D] (written): dL/dq,
 *       dL/dk, dL/dv in the same dtype and shard-major layout as the inputs.
 *   workspace (device, caller-owned, 16-byte aligned, read and written):
 *       workspace_bytes >= the size ra_backward_workspace reports for the
 *       shape.  Holds the per-row terms delta; nothing in it outlives the
 *       call.
 * The pages name training as the use of the method (1M-token LLM training;
 * end-to-end training throughput under Striped Attention; PyTorch's
 * context_parallel replacing scaled dot-product attention when training)
 * but do not write the backward out.  It is the chain rule of the forward's
 * definition.  For query row t, visible key u, P_tu = exp(scale q_t.k_u -
 * lse_t):
 *   delta_t = dout_t . out_t
 *   dv_u = sum_t P_tu dout_t          dS_tu = P_tu (dout_t . v_u - delta_t)
 *   dq_t = scale sum_u dS_tu k_u      dk_u = scale sum_t dS_tu q_t
 * and a key/value head's gradient sums over the query heads that read it.
 * The fold follows the ring: dq of query shard i accumulates over key/value
 * shards j = (i - s) mod N in the forward's order (entered at shard N-1 on
 * the tensor-core path when the blocks the query tiles in flight read at
 * once exceed the L2, as in ra_forward), and the accumulators of dk and dv
 * of shard j travel with the block round the ring in its cyclic order,
 * entering it at device 0 (ra_plan_backward lists the order).
 * Shards and tiles without a visible pair are skipped.
 * Kernels: the tcgen05 tensor-core backward for bf16, D in {64, 128} (any Sb
 * for contiguous and striped shards, Sb % 256 == 0 for zigzag), else the fp32
 * SIMT backward (f32 or bf16, D <= 128).  ra_backward_ex chooses explicitly.
 * Neither uses atomics: for fixed inputs the gradients are the same bits on
 * every call.
 * An empty problem (B == 0 or S == 0) is a no-op, as in ra_forward; every
 * pointer may then be NULL and workspace_bytes 0.
 * Errors: as ra_forward; RA_ERR_CAPACITY when workspace_bytes is too small;
 * RA_ERR_UNSUPPORTED for D > 128.
 */
int ra_backward(const void* q, const void* k, const void* v, const void* out, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, void* workspace,
                int64_t workspace_bytes, int B, int Hq, int Hkv, int64_t S, int D, int N,
                int causal, int striped, float scale, int dtype, void* stream);

/* ra_backward with an explicit kernel choice (RA_KERNEL_*).  RA_KERNEL_TC
 * returns RA_ERR_UNSUPPORTED outside its envelope. */
int ra_backward_ex(const void* q, const void* k, const void* v, const void* out,
                   const float* lse, const void* dout, void* dq, void* dk, void* dv,
                   void* workspace, int64_t workspace_bytes, int B, int Hq, int Hkv, int64_t S,
                   int D, int N, int causal, int striped, float scale, int dtype, int kernel,
                   void* stream);

/* ra_backward_workspace (host only): bytes of workspace ra_backward needs for
 * the shape: 4*B*Hq*S for delta, rounded up to 256 (D does not enter).
 * Errors: RA_ERR_INVALID_ARG (negative B or S, non-positive Hq or D, or a
 * null bytes pointer).  An empty problem needs 0 bytes. */
int ra_backward_workspace(int B, int Hq, int64_t S, int D, int64_t* bytes);

/*
 * ra_watchdog_selftest_backward: the failure-detection self test of one
 * backward tensor-core kernel (which = 0: the dq kernel, 1: the dk/dv
 * kernel), the counterpart of ra_watchdog_selftest.  Arguments as
 * ra_backward (bf16, tensor-core shapes) plus timeout_cycles (1e5 .. 4e9
 * SM clock cycles): the kernel's first K (dq) or Q (dk/dv) tile copy is never
 * issued and every wait is bounded by timeout_cycles, so the waits that
 * depend on it run out; the kernel records RA_ERR_TIMEOUT in the device
 * status word, lets its copies and MMAs in flight finish, frees its tensor
 * memory and returns.  The gradients are left undefined.  Returns RA_OK once
 * enqueued; ra_check(stream) then reports RA_ERR_TIMEOUT.
 * Errors: as ra_backward; RA_ERR_INVALID_ARG for timeout_cycles out of range,
 * `which` not 0 or 1 or an empty problem; RA_ERR_UNSUPPORTED outside the tensor-core shapes.
 */
int ra_watchdog_selftest_backward(const void* q, const void* k, const void* v, const void* out,
                                  const float* lse, const void* dout, void* dq, void* dk,
                                  void* dv, void* workspace, int64_t workspace_bytes, int B,
                                  int Hq, int Hkv, int64_t S, int D, int N, int causal,
                                  int striped, float scale, int64_t timeout_cycles, int which,
                                  void* stream);

/*
 * ra_check: synchronise `stream`, then read and clear this device's status
 * word.  Returns RA_OK, RA_ERR_TIMEOUT, RA_ERR_BOUNDS or RA_ERR_CUDA (the
 * synchronisation itself failed; the CUDA error string is kept for
 * ra_strerror(RA_ERR_CUDA)).
 */
int ra_check(void* stream);

/*
 * ra_forward_noalloc: ra_forward for callers that cannot allocate device
 * memory.  The pages describe nothing like it; it exists because some
 * programs must not call cudaMalloc while they run attention: a server that
 * reserved all device memory for its own pool at start-up, a framework whose
 * caching allocator owns the GPU, or latency-critical code that cannot take
 * cudaMalloc's device-wide synchronisation or its out-of-memory failure.
 * ra_forward allocates a 4 KiB scratch block on its first tensor-core call on
 * a device; this entry point allocates nothing.  Its scratch, the kernel's
 * work-queue counter, lives in a 256-byte static __device__ array that every
 * device loading the library holds until the process exits.
 *   Arguments, layouts and results are those of ra_forward_ex with
 *   dtype = RA_BF16 and RA_KERNEL_TC (the work-queue form: the stream-K form
 *   ra_forward picks for few-item non-causal problems takes scratch); only
 *   the tensor-core kernel's shapes are accepted (D in {64, 128}; S/N a
 *   multiple of 256 for zigzag).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call outside CUDA-graph stream
 *   capture.  Each call zeroes the counter on `stream` before its kernel.
 *   All calls share the one array: calls whose kernels may overlap on the GPU
 *   (different streams without ordering between them) race on it.  Order
 *   them on one stream or with events.
 * An empty problem is a no-op, as in ra_forward.
 * Errors: as ra_forward; RA_ERR_UNSUPPORTED outside the tensor-core shapes;
 * RA_ERR_CAPACITY when the scratch the call needs exceeds the array (one
 * 32-bit counter, so at most 2^31 work items).
 */
int ra_forward_noalloc(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                       int Hq, int Hkv, int64_t S, int D, int N, int causal, int striped,
                       float scale, void* stream);

/* Human-readable text for a status code (static storage). */
const char* ra_strerror(int code);

/* Query/key tile sizes of the tensor-core kernel (both 128). */
int ra_tile_config(int* tq, int* tk);

/* Library version as major*10000 + minor*100 + patch. */
int ra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
