// Tensor-core (tcgen05) ring-attention forward kernel for sm_103a, bf16 in,
// fp32 accumulate.
//
// What it computes (the pages' method): each 128-row query tile of shard i
// folds the key/value shards j = (i - s) mod N, s = 0..N-1, one 128-key tile
// at a time, into a running row max m, running normaliser l and an
// unnormalised numerator O held in tensor memory; O / l is written at the end
// ("Ring Attention" glossary page, "Como funciona a atencao em anel";
// aiunderstanding.org, "Approfondimento tecnico").  Whole shards and key tiles
// with no visible pair are never visited (the schedule in schedule.cuh).
//
// How (B300 design):
//  * Persistent grid, one CTA per SM (512 TMEM columns, ~193 KB smem).  A CTA
//    works on items of two query tiles ("slots") that share each K/V tile.
//  * warp 0, lane 0 -- TMA producer: Q tiles once per item, then K and V
//    tiles into a ring of smem stages (128B-swizzled, 2 boxes of 64 columns).
//  * lane 0 of warps 1 and 3 -- MMA issuers, one per slot: S_t = Q_t K^T (SS,
//    M=128 N=128 K=16 steps) into TMEM, and O_t += P_t V (P read from TMEM, V
//    MN-major from smem).  A token passed between them keeps the pipe order
//    PV_0(n-1) S_0(n) | PV_1(n-1) S_1(n) | ...: while one softmax warpgroup
//    works, the tensor core runs the other slot's MMAs, and each issuer's
//    waits overlap the other issuer's MMA issue.
//  * warp 2 owns the TMEM allocation.
//  * warps 4-7 / 8-11 -- softmax for slot 0 / 1, one thread per query row
//    (row r = TMEM lane r): load the S row, mask the diagonal tile, update
//    the running max, exp2, write P (bf16) over the S columns, and rescale
//    O only when the max grew by more than 2^8 (the fold stays exact: the
//    same stale max is used for numerator and normaliser).  They also run
//    the epilogue O / l and lse = m + ln l.
//  * Every mbarrier wait is bounded; on time-out the kernel records
//    kStatusTimeout in the device status word, drains its in-flight copies
//    and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "ra.h"
#include "schedule.cuh"
#include "tmap.h"
#include "waits.cuh"

namespace ra {
namespace tc {

constexpr int kT = 128;             // query and key tile size
constexpr int kThreads = 384;       // 12 warps
// Bounded waits count SM clock cycles (4e9 cycles is 2 s at 2 GHz, longer at lower clocks).
constexpr long long kTimeoutCycles = 4000000000ll;
constexpr long long kDrainCycles = 400000000ll;
// Register split: 384 threads launched at 168 registers (64512 in total);
// warpgroup 0 (producer, MMA, TMEM owner) drops to 80, the two softmax
// warpgroups rise to 208: 128*80 + 256*208 = 63488 <= 64512.  The softmax
// writes P and rescales O 16 TMEM columns at a time so that its loop, which
// holds the S row in 128 registers, does not spill at 208.
constexpr uint32_t kRegsOther = 80, kRegsSoftmax = 208;

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kT * D * 2;
    static constexpr int kStages = (D == 128) ? 4 : 8;
    static constexpr int kBoxes = D / 64;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
    // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_lo[2], p_hi[2],
    // o_full[2], o_empty[2], drain[2], token[2], item_full[2], item_empty[2]
    static constexpr int kNumBars = 2 + 2 * kStages + 18;
    static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 16 + 1024;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColO0 = 256, kColO1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
    // barrier indices
    static constexpr int bQFull = 0, bQEmpty = 1, bKVFull = 2, bKVEmpty = 2 + kStages,
                         bSFull = 2 + 2 * kStages, bPLo = bSFull + 2, bPHi = bPLo + 2,
                         bOFull = bPHi + 2,
                         bOEmpty = bOFull + 2, bDrain = bOEmpty + 2, bToken = bDrain + 2,
                         bItemFull = bToken + 2, bItemEmpty = bItemFull + 2;
    // readers of each published item: two MMA issuers + eight softmax warps
    static constexpr uint32_t kItemReaders = 10;
};

struct Params {
    ItemGeom G;
    int64_t S;
    int Sb;
    int rem;  // rows of each shard's last tile (128 unless Sb % 128 != 0)
    float sl2;  // scale * log2(e)
    __nv_bfloat16* out;
    float* lse;
    unsigned int* status;
    int32_t* log;
    int32_t* counts;
    int max_entries;
    unsigned int* work;  // item counter, zero at launch: CTAs take items in order
    long long timeout_cycles;  // self test only: limit of every bounded wait
    // Ring step only (STEP kernels): the buffers hold query shard step_i and
    // key/value block step_j alone (S = Sb rows per (b, h) slice); the items
    // cover the shard's query tiles, `ring` is the real ring whose masks apply,
    // and the epilogue folds the block's partial into the running state.
    RingGeom ring;
    int step_i, step_j, step_s;
    int step_first, step_last;
    float* state_o;    // [B*Hq*Sb, D] running normalised output (fp32)
    float* state_lse;  // [B*Hq*Sb] running log-sum-exp (natural log)
    // Stream-K launches only (non-causal problems with one to two items per
    // SM, every item folding fold_len key tiles): CTA c takes the c-th equal,
    // contiguous range of the flattened (item, fold position) space instead of
    // items from the queue, so the last wave leaves no SM idle.  An item cut
    // between CTAs c and c+1 runs as a head segment [0, p) at the end of c's
    // range and a tail segment [p, fold_len) at the start of c+1's.  The tail
    // writes its partial (O/l and lse, fp32) to part_o / part_lse and raises
    // its warp's flag; the head, which finishes later, waits for the flag and
    // combines the partial with its own O and l by the log-sum-exp weighting.
    long long n_work;          // work values >= n_work end a CTA's loop
    int fold_len;
    float* part_o;             // [n_items][2 slots][D/4 chunks][128 rows] float4
    float* part_lse;           // [n_items][2 slots][128 rows]
    unsigned int* part_flag;   // [n_items][2 slots][4 warps], zero at launch
};

enum Mode : int { kModeRing = 0, kModeStep = 1, kModeStreamK = 2, kModeRingFromLast = 3 };

// The walk type of a mode: kModeRingFromLast enters every query shard's ring
// at block N-1 (ring_entry), the other modes take the ring order.
template <int MODE>
using WalkT =
    typename std::conditional<MODE == kModeRingFromLast, TileWalkFromLast, TileWalk>::type;

// A work value: an item index, or in stream-K launches an item and the range
// [b, e) of its fold positions, packed as item << 32 | b << 16 | e.
struct Work {
    long long item;
    int b, e;
};

// The fold list of an item: every ring step (TileWalk), the key tiles of
// the one block a ring step holds, or fold positions [b, e) of a stream-K
// segment (non-causal: position s*nt + kt is key tile kt of shard (i - s)).
template <int MODE>
__device__ __forceinline__ void walk_start(WalkT<MODE>& w, const ItemGeom& G, const Params& p,
                                           const Item& it, const Work& wk) {
    if constexpr (MODE == kModeStep) {
        w.s = p.step_s;
        w.j = p.step_j;
        w.kt = 0;
        int nk0, nk1, d;
        shard_span(p.ring, p.step_i, p.step_j, it.qt[0], &nk0, &d);
        shard_span(p.ring, p.step_i, p.step_j, it.qt[1], &nk1, &d);
        w.nk = nk0 > nk1 ? nk0 : nk1;
    } else if constexpr (MODE == kModeStreamK) {
        const int nt = G.rg.nt;
        w.s = wk.b / nt;
        w.kt = wk.b % nt;
        w.nk = wk.e;  // the end position
        w.j = it.i - w.s;
        if (w.j < 0) w.j += G.rg.N;
    } else {
        (void)wk;
        w.start(G.rg, it);
    }
}
template <int MODE>
__device__ __forceinline__ bool walk_done(const WalkT<MODE>& w, const ItemGeom& G) {
    if constexpr (MODE == kModeStep) return w.kt >= w.nk;
    else if constexpr (MODE == kModeStreamK) return w.s * G.rg.nt + w.kt >= w.nk;
    else return w.done(G.rg);
}
template <int MODE>
__device__ __forceinline__ void walk_next(WalkT<MODE>& w, const ItemGeom& G, const Item& it) {
    if constexpr (MODE == kModeStep) {
        ++w.kt;
    } else if constexpr (MODE == kModeStreamK) {
        if (++w.kt >= G.rg.nt) {
            w.kt = 0;
            ++w.s;
            w.j = it.i - w.s;
            if (w.j < 0) w.j += G.rg.N;
        }
    } else {
        w.next(G.rg, it);
    }
}
template <int MODE>
__device__ __forceinline__ Work decode_work(long long v) {
    Work wk;
    if constexpr (MODE == kModeStreamK) {
        wk.item = v >> 32;
        wk.b = (int)((v >> 16) & 0xffff);
        wk.e = (int)(v & 0xffff);
    } else {
        wk.item = v;
        wk.b = wk.e = 0;
    }
    return wk;
}

// MODE: kModeRing (the whole ring, items from the dynamic queue),
// kModeRingFromLast (the same, every query shard entering at block N-1),
// kModeStep (one step of a ring whose devices are separate processes) or
// kModeStreamK (fixed contiguous work ranges per CTA; see Params).
template <int D, bool LOG, bool SELFTEST, bool RAGGED, int MODE = kModeRing>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const Params p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile long long* item_slot = reinterpret_cast<volatile long long*>(tmem_slot + 4);  // [2]
    auto bar = [&](int idx) -> uint32_t { return base + C::kBarOff + idx * 8; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ItemGeom& G = p.G;
    // limit of every bounded wait (the failure-detection self test uses a short one)
    const long long wlim = SELFTEST ? p.timeout_cycles : kTimeoutCycles;

    if (tid == 0) {
        mbar_init(bar(C::bQFull), 1);
        mbar_init(bar(C::bQEmpty), 2);  // one commit per MMA issuer
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::bKVFull + s), 1);
            mbar_init(bar(C::bKVEmpty + s), 2);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::bSFull + t), 1);
            mbar_init(bar(C::bPLo + t), 4);
            mbar_init(bar(C::bPHi + t), 4);
            mbar_init(bar(C::bOFull + t), 1);
            mbar_init(bar(C::bOEmpty + t), 4);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::bDrain + t), 1);
            mbar_init(bar(C::bToken + t), 1);
            mbar_init(bar(C::bItemFull + t), 1);
            mbar_init(bar(C::bItemEmpty + t), C::kItemReaders);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Work items are handed out dynamically in their longest-first order: the
    // producer takes the next index from the global counter one item ahead and
    // publishes it in a two-entry shared ring; every role reads it from there.
    // An index >= n_items ends the CTA's loop.
    constexpr bool STEP = MODE == kModeStep, STREAMK = MODE == kModeStreamK;
    auto read_item = [&](int k, bool& ok) -> long long {
        ok = wait_bar(bar(C::bItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status, wlim);
        return ok ? item_slot[k & 1] : p.n_work;
    };
    if (warp < 4) regs_dec<kRegsOther>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            uint32_t kv_pos = 0, q_loads = 0;
            int k = 0;
            bool ok = true;
            auto publish = [&](int kk, long long v) -> bool {
                if (kk >= 2 && !wait_bar(bar(C::bItemEmpty + (kk & 1)), ((kk >> 1) - 1) & 1,
                                         abort_flag, p.status, wlim))
                    return false;
                item_slot[kk & 1] = v;
                mbar_arrive(bar(C::bItemFull + (kk & 1)));
                return true;
            };
            // stream-K: this CTA's contiguous range of (item, fold position)
            const long long total = STREAMK ? G.n_items * (long long)p.fold_len : 0;
            long long sk_cur = STREAMK ? total * blockIdx.x / gridDim.x : 0;
            const long long sk_end = STREAMK ? total * (blockIdx.x + 1) / gridDim.x : 0;
            auto next_work = [&]() -> long long {
                if constexpr (STREAMK) {
                    if (sk_cur >= sk_end) return p.n_work;
                    const long long itm = sk_cur / p.fold_len;
                    const int b = (int)(sk_cur % p.fold_len);
                    const long long left = sk_end - sk_cur;
                    const int e = (left < p.fold_len - b) ? b + (int)left : p.fold_len;
                    sk_cur += e - b;
                    return (itm << 32) | ((long long)b << 16) | e;
                } else {
                    return (long long)atomicAdd(p.work, 1u);
                }
            };
            long long item = next_work();
            ok = publish(0, item);
            for (; ok && item < p.n_work; ++k) {
                const long long next = next_work();
                if (!(ok = publish(k + 1, next))) break;
                const Work wk = decode_work<MODE>(item);
                const Item it = decode_item(G, wk.item);
                item = next;
                if (k > 0 && !(ok = wait_bar(bar(C::bQEmpty), (k - 1) & 1, abort_flag, p.status, wlim)))
                    break;
                mbar_arrive_expect_tx(bar(C::bQFull), 2 * C::kTileBytes);
                ++q_loads;
                for (int t = 0; t < 2; ++t) {
                    const int row = (int)((int64_t)(it.b * G.Hq + it.h[t]) * p.S +
                                          (int64_t)it.i * p.Sb + (int64_t)it.qt[t] * kT);
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        tma_load_2d(base + C::kQOff + t * C::kTileBytes + bx * (kT * 128), &tm_q,
                                    bx * 64, row, bar(C::bQFull), pol_q);
                }
                const int64_t kvrow0 = (int64_t)(it.b * G.Hkv + it.kvh) * p.S;
                WalkT<MODE> w;
                for (walk_start<MODE>(w, G, p, it, wk); !walk_done<MODE>(w, G) && ok;
                     walk_next<MODE>(w, G, it)) {
                    // a ring step's buffer holds only the block it folds
                    const int64_t jrow = STEP ? 0 : (int64_t)w.j * p.Sb;
                    const int row = (int)(kvrow0 + jrow + (int64_t)w.kt * kT);
                    for (int kv = 0; kv < 2; ++kv) {
                        if (SELFTEST && kv_pos == 0) {  // self test: nothing ever signals stage 0
                            ++kv_pos;
                            continue;
                        }
                        const uint32_t st = kv_pos % C::kStages, use = kv_pos / C::kStages;
                        if (use > 0 && !(ok = wait_bar(bar(C::bKVEmpty + st), (use - 1) & 1,
                                                       abort_flag, p.status, wlim)))
                            break;
                        mbar_arrive_expect_tx(bar(C::bKVFull + st), C::kTileBytes);
                        const CUtensorMap* tm = kv ? &tm_v : &tm_k;
                        for (int bx = 0; bx < C::kBoxes; ++bx)
                            tma_load_2d(base + C::kKVOff + st * C::kTileBytes + bx * (kT * 128), tm,
                                        bx * 64, row, bar(C::bKVFull + st), pol_kv);
                        ++kv_pos;
                    }
                }
                if (!ok) break;
            }
            if (!ok) {
                // let every copy that may still be in flight land before exit
                if (q_loads > 0) drain_wait(bar(C::bQFull), (q_loads - 1) & 1, kDrainCycles);
                const uint32_t first = kv_pos > (uint32_t)C::kStages ? kv_pos - C::kStages : 0;
                for (uint32_t pos = first; pos < kv_pos; ++pos)
                    drain_wait(bar(C::bKVFull + pos % C::kStages), (pos / C::kStages) & 1, kDrainCycles);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA issuers
        // Lane 0 of warp 1 issues slot 0's MMAs, lane 0 of warp 3 slot 1's.  A
        // token (two mbarriers) makes them take turns block by block, so the
        // tensor pipe still sees PV_0 S_0 | PV_1 S_1 | PV_0 S_0 ... in order,
        // while each issuer's own waits overlap the other's issue.
        if (lane == 0) {
            const int t = (warp == 1) ? 0 : 1;
            constexpr uint32_t idesc_s = make_idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_o = make_idesc_bf16(128, D, false, true);
            const uint32_t qa = base + C::kQOff + t * C::kTileBytes;
            const uint32_t s_tm = tmem + (t ? C::kColS1 : C::kColS0);
            const uint32_t o_tm = tmem + (t ? C::kColO1 : C::kColO0);
            const uint64_t dq = make_sdesc(qa, 16, 1024, kLayoutSW128);
            auto issue_s = [&](uint32_t stK) {
                const uint64_t dk =
                    make_sdesc(base + C::kKVOff + stK * C::kTileBytes, 16, 1024, kLayoutSW128);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // start address advances in 16-byte units inside the descriptor
                    const uint32_t off16 = ((kk / 4) * (kT * 128) + (kk % 4) * 32) >> 4;
                    umma_ss(s_tm, dq + off16, dk + off16, idesc_s, kk > 0);
                }
            };
            // O += P[:, 64h : 64h+64] V[64h : 64h+64, :]  (keys half h)
            auto issue_pv_half = [&](uint32_t stV, int h, bool acc) {
                const uint64_t dv = make_sdesc(base + C::kKVOff + stV * C::kTileBytes, kT * 128,
                                               1024, kLayoutSW128);
#pragma unroll
                for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                    umma_ts(o_tm, s_tm + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), idesc_o,
                            (kk > 0 || acc) ? 1u : 0u);
            };
            // P of the previous key tile arrives in two halves; the first half's
            // MMAs run while the softmax still computes the second half.  The
            // caller has already waited for the first half.
            auto issue_pv = [&](uint32_t stV, bool acc, uint32_t g) -> bool {
                issue_pv_half(stV, 0, acc);
                if (!wait_bar(bar(C::bPHi + t), g & 1, abort_flag, p.status, wlim)) return false;
                tc_fence_after();
                issue_pv_half(stV, 1, acc);
                return true;
            };
            // block counter: slot 0 issues its block b after slot 1's block b-1,
            // slot 1 issues block b after slot 0's block b
            uint32_t bc = 0;
            auto take_turn = [&]() -> bool {
                if (t == 0) return bc == 0 || wait_bar(bar(C::bToken + 0), (bc - 1) & 1, abort_flag, p.status, wlim);
                return wait_bar(bar(C::bToken + 1), bc & 1, abort_flag, p.status, wlim);
            };
            auto pass_turn = [&]() {
                mbar_arrive(bar(C::bToken + (t == 0 ? 1 : 0)));
                ++bc;
            };
            uint32_t kv_pos = 0, gt = 0;
            int k = 0;
            bool ok = true;
            for (;; ++k) {
                const long long item = read_item(k, ok);
                if (ok) mbar_arrive(bar(C::bItemEmpty + (k & 1)));
                if (!ok || item >= p.n_work) break;
                const Work wk = decode_work<MODE>(item);
                const Item it = decode_item(G, wk.item);
                if (!(ok = wait_bar(bar(C::bQFull), k & 1, abort_flag, p.status, wlim))) break;
                WalkT<MODE> w;
                uint32_t n = 0;
                for (walk_start<MODE>(w, G, p, it, wk); !walk_done<MODE>(w, G);
                     walk_next<MODE>(w, G, it), ++n) {
                    const uint32_t stK = kv_pos % C::kStages;
                    if (!(ok = wait_bar(bar(C::bKVFull + stK), (kv_pos / C::kStages) & 1,
                                        abort_flag, p.status, wlim)))
                        break;
                    uint32_t stV = 0;
                    if (n > 0) {
                        const uint32_t vp = kv_pos - 1;
                        stV = vp % C::kStages;
                        if (!(ok = wait_bar(bar(C::bKVFull + stV), (vp / C::kStages) & 1,
                                            abort_flag, p.status, wlim)))
                            break;
                        if (!(ok = wait_bar(bar(C::bPLo + t), (gt - 1) & 1, abort_flag,
                                            p.status, wlim)))
                            break;
                        if (n == 1 && k > 0 &&
                            !(ok = wait_bar(bar(C::bOEmpty + t), (k - 1) & 1, abort_flag,
                                            p.status, wlim)))
                            break;
                    }
                    if (!(ok = take_turn())) break;
                    tc_fence_after();
                    if (n > 0) {
                        if (!(ok = issue_pv(stV, n > 1, gt - 1))) break;
                        umma_commit(bar(C::bKVEmpty + stV));
                    }
                    issue_s(stK);
                    pass_turn();
                    umma_commit(bar(C::bSFull + t));
                    umma_commit(bar(C::bKVEmpty + stK));
                    kv_pos += 2;
                    ++gt;
                }
                if (!ok) break;
                if (STEP && n == 0) {
                    // no tile of this block is visible to the item: no MMA reads
                    // its Q tile or writes its O, so release both at once
                    mbar_arrive(bar(C::bQEmpty));
                    mbar_arrive(bar(C::bOFull + t));
                    continue;
                }
                umma_commit(bar(C::bQEmpty));  // every S MMA of this slot and item is issued
                const uint32_t vp = kv_pos - 1, stV = vp % C::kStages;
                if (!(ok = wait_bar(bar(C::bKVFull + stV), (vp / C::kStages) & 1, abort_flag,
                                    p.status, wlim)))
                    break;
                if (!(ok = wait_bar(bar(C::bPLo + t), (gt - 1) & 1, abort_flag, p.status, wlim)))
                    break;
                if (n == 1 && k > 0 &&
                    !(ok = wait_bar(bar(C::bOEmpty + t), (k - 1) & 1, abort_flag, p.status, wlim)))
                    break;
                if (!(ok = take_turn())) break;
                tc_fence_after();
                if (!(ok = issue_pv(stV, n > 1, gt - 1))) break;
                pass_turn();
                umma_commit(bar(C::bOFull + t));
                umma_commit(bar(C::bKVEmpty + stV));
            }
            if (!ok) {
                *abort_flag = 1;
                umma_commit(bar(C::bDrain + t));
                drain_wait(bar(C::bDrain + t), 0, kDrainCycles);
            }
        }
    } else if (warp < 4) {
        // warp 2: TMEM owner
    } else {
        // ------------------------------------------------------------ softmax
        regs_inc<kRegsSoftmax>();
        const int t = (warp - 4) >> 2;
        const int r = tid - 128 * (1 + t);  // query row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_tm = tmem + lane_off + (t ? C::kColS1 : C::kColS0);
        const uint32_t o_tm = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
        const float sl2 = p.sl2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint32_t gt = 0;
        int k = 0;
        bool ok = true;
        for (;; ++k) {
            const long long item = read_item(k, ok);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bItemEmpty + (k & 1)));
            if (item >= p.n_work) break;
            const Work wk = decode_work<MODE>(item);
            const Item it = decode_item(G, wk.item);
            const int qt = t ? it.qt[1] : it.qt[0];
            const int hq = t ? it.h[1] : it.h[0];  // query head of this slot
            const bool valid = (t == 0) || it.valid1;
            float m_used = -INFINITY, l = 0.f;
            int n_logged = 0;
            WalkT<MODE> w;
            uint32_t n = 0;
            for (walk_start<MODE>(w, G, p, it, wk); !walk_done<MODE>(w, G);
                 walk_next<MODE>(w, G, it), ++n, ++gt) {
                const int kind = STEP ? fold_kind(p.ring, p.step_i, w.j, qt, w.kt)
                                      : fold_kind(G.rg, it.i, w.j, qt, w.kt);
                ok = wait_bar(bar(C::bSFull + t), gt & 1, abort_flag, p.status, wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                if (kind == kNone) {
                    uint32_t z[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] = 0u;
                    tmem_st32(s_tm + 0, z);
                    tmem_st32(s_tm + 32, z);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::bPLo + t));
                } else {
                    uint32_t sr[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + c * 32, sr[c]);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
                    // visible iff col <= lim: the diagonal masks, and on a shard's
                    // last (partial) key tile the columns past the shard's end
                    int lim = (kind == kIncl) ? r : (kind == kStrict) ? r - 1 : kT - 1;
                    if (RAGGED && w.kt == G.rg.nt - 1 && p.rem - 1 < lim) lim = p.rem - 1;
                    if (lim < kT - 1) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (c * 32 + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
                    }
                    // row max: four independent chains of three-input max
                    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) {
                            mx0 = max3f(mx0, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
                            mx1 = max3f(mx1, __uint_as_float(sr[c][e + 2]), __uint_as_float(sr[c][e + 3]));
                            mx2 = max3f(mx2, __uint_as_float(sr[c][e + 4]), __uint_as_float(sr[c][e + 5]));
                            mx3 = max3f(mx3, __uint_as_float(sr[c][e + 6]), __uint_as_float(sr[c][e + 7]));
                        }
                    }
                    const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3));
                    const float m_new = fmaxf(m_used, mx);
                    // rescale only when the max grew by more than 2^8 (in exp2 units)
                    const bool need = (m_new - m_used) * sl2 > 8.0f;
                    if (__any_sync(0xffffffffu, need)) {
                        float alpha = 1.f;
                        if (need) {
                            alpha = ex2_approx((m_used - m_new) * sl2);
                            m_used = m_new;
                        }
                        l *= alpha;
                        if (n > 0) {
                            // 16 columns at a time: the S row is live in 128 registers here
                            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                            for (int c = 0; c < D / 16; ++c) {
                                uint32_t o[16];
                                tmem_ld16(o_tm + c * 16, o);
                                tmem_wait_ld();
                                reg_fence(o);
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    float lo, hi;
                                    f2_unpack(f2_mul(f2_pack_u(o[e], o[e + 1]), a2), lo, hi);
                                    o[e] = __float_as_uint(lo);
                                    o[e + 1] = __float_as_uint(hi);
                                }
                                tmem_st16(o_tm + c * 16, o);
                            }
                        }
                    }
                    const float mb = (m_used == -INFINITY) ? 0.f : m_used * sl2;
                    const uint64_t nmb2 = f2_pack(-mb, -mb);
                    uint64_t acc0 = 0, acc1 = 0;  // packed fp32 pairs (0.0f, 0.0f)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {  // keys [32c, 32c + 32) -> P columns [16c, 16c + 16)
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            const uint64_t x01 = f2_fma(f2_pack_u(sr[c][e], sr[c][e + 1]), sl2x2, nmb2);
                            const uint64_t x23 = f2_fma(f2_pack_u(sr[c][e + 2], sr[c][e + 3]), sl2x2, nmb2);
                            float a0, a1, a2, a3;
                            f2_unpack(x01, a0, a1);
                            f2_unpack(x23, a2, a3);
                            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
                            const float p2 = ex2_approx(a2), p3 = ex2_approx(a3);
                            acc0 = f2_add(acc0, f2_pack(p0, p1));
                            acc1 = f2_add(acc1, f2_pack(p2, p3));
                            pk[e / 2] = pack_bf16x2(p0, p1);
                            pk[e / 2 + 1] = pack_bf16x2(p2, p3);
                        }
                        tmem_st16(s_tm + 16 * c, pk);
                        if (c == 1) {  // first 64 keys of P are in TMEM: let P.V start on them
                            tmem_wait_st();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar(C::bPLo + t));
                        }
                    }
                    float s0, s1, s2, s3;
                    f2_unpack(f2_add(acc0, acc1), s0, s1);
                    (void)s2;
                    (void)s3;
                    l += s0 + s1;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::bPHi + t));
                if (LOG && valid && kind != kNone && r == 0) {
                    const int64_t unit =
                        ((int64_t)(it.b * G.Hq + hq) * G.rg.N + it.i) * G.rg.nt + qt;
                    if (n_logged < p.max_entries) {
                        int32_t* e = p.log + (unit * p.max_entries + n_logged) * 4;
                        e[0] = w.s;
                        e[1] = w.j;
                        e[2] = w.kt;
                        e[3] = kind;
                    } else {
                        atomicOr(p.status, kStatusBounds);
                    }
                    ++n_logged;
                }
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            ok = wait_bar(bar(C::bOFull + t), k & 1, abort_flag, p.status, wlim);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            if (STEP && valid) {
                // Fold this block's partial (O/l, lse_b) into the running state
                // (O_s, lse_s) by the log-sum-exp weighting, in exp2 units:
                //   lse = log2(2^a + 2^b),  O = 2^(a-lse) O_s + 2^(b-lse) O/l.
                // Rows this block leaves empty (l = 0) keep the state.
                const int64_t row = (int64_t)(it.b * G.Hq + hq) * p.S + (int64_t)qt * kT + r;
                const bool row_ok = !RAGGED || qt < G.rg.nt - 1 || r < p.rem;
                constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.69314718055994531f;
                const float b2 = (l > 0.f) ? m_used * sl2 + lg2_approx(l) : -INFINITY;
                const float a2 = (!p.step_first && row_ok) ? p.state_lse[row] * kLog2e : -INFINITY;
                const float mx = fmaxf(a2, b2);
                float cs = 0.f, cp = 0.f, lse_n = -INFINITY;
                if (mx > -INFINITY) {
                    const float ws = ex2_approx(a2 - mx), wp = ex2_approx(b2 - mx);
                    const float den = ws + wp;
                    cs = ws / den;
                    cp = (l > 0.f) ? wp / den / l : 0.f;
                    lse_n = (mx + lg2_approx(den)) * kLn2;
                }
                const bool use_o = l > 0.f;
                float4* srow = reinterpret_cast<float4*>(p.state_o + row * D);
                uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(o_tm + c * 32, o);  // warp-collective: every lane loads
                    tmem_wait_ld();
                    reg_fence(o);
                    float nv[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) nv[e] = use_o ? cp * __uint_as_float(o[e]) : 0.f;
                    if (!p.step_first && row_ok) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 sv = srow[c * 8 + e];
                            nv[4 * e] = fmaf(cs, sv.x, nv[4 * e]);
                            nv[4 * e + 1] = fmaf(cs, sv.y, nv[4 * e + 1]);
                            nv[4 * e + 2] = fmaf(cs, sv.z, nv[4 * e + 2]);
                            nv[4 * e + 3] = fmaf(cs, sv.w, nv[4 * e + 3]);
                        }
                    }
                    if (row_ok) {
                        if (p.step_last) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                orow[c * 4 + e] = make_uint4(
                                    pack_bf16x2(nv[8 * e], nv[8 * e + 1]),
                                    pack_bf16x2(nv[8 * e + 2], nv[8 * e + 3]),
                                    pack_bf16x2(nv[8 * e + 4], nv[8 * e + 5]),
                                    pack_bf16x2(nv[8 * e + 6], nv[8 * e + 7]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                srow[c * 8 + e] = make_float4(nv[4 * e], nv[4 * e + 1],
                                                              nv[4 * e + 2], nv[4 * e + 3]);
                        }
                    }
                }
                if (row_ok) {
                    if (!p.step_last) p.state_lse[row] = lse_n;
                    else if (p.lse) p.lse[row] = lse_n;
                }
            } else if (STREAMK && valid && !(wk.b == 0 && wk.e == p.fold_len)) {
                // A segment of an item cut between two CTAs (see Params).
                const int64_t row = (int64_t)(it.b * G.Hq + hq) * p.S + (int64_t)it.i * p.Sb +
                                    (int64_t)qt * kT + r;
                const bool row_ok = !RAGGED || qt < G.rg.nt - 1 || r < p.rem;
                constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.69314718055994531f;
                const int64_t blk = wk.item * 2 + t;  // the tail's partial of this slot
                // column-chunk-major: float4 chunk cc of row r at [blk][cc][r], so
                // a warp's 32 rows move 512 contiguous bytes per chunk
                float4* pblk = reinterpret_cast<float4*>(p.part_o) + blk * (D / 4) * kT + r;
                unsigned int* flag = p.part_flag + blk * 4 + (warp & 3);
                const bool use_o = l > 0.f;
                const float lse_own = use_o ? (m_used * sl2 + lg2_approx(l)) * kLn2 : -INFINITY;
                if (wk.b > 0) {
                    // tail segment: write the partial (O/l, lse), then raise the flag
                    const float inv_l = use_o ? 1.f / l : 0.f;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_tm + c * 32, o);  // warp-collective: every lane loads
                        tmem_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            pblk[(c * 8 + e) * kT] =
                                make_float4(__uint_as_float(o[4 * e]) * inv_l,
                                            __uint_as_float(o[4 * e + 1]) * inv_l,
                                            __uint_as_float(o[4 * e + 2]) * inv_l,
                                            __uint_as_float(o[4 * e + 3]) * inv_l);
                    }
                    p.part_lse[blk * kT + r] = lse_own;
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicExch(flag, 1u);
                } else {
                    // head segment, at the end of the previous CTA's range: the
                    // tail ran at the start of the next CTA's, so its flag is
                    // normally up already.  The wait is bounded all the same.
                    bool have = true;
                    if (lane == 0) {
                        const long long t0 = clock64();
                        while (atomicAdd(flag, 0u) == 0u) {
                            if (clock64() - t0 > wlim) {
                                atomicOr(p.status, kStatusTimeout);
                                have = false;
                                break;
                            }
                        }
                    }
                    have = __shfl_sync(0xffffffffu, have ? 1 : 0, 0) != 0;
                    __threadfence();
                    const float lse_tail = have ? __ldcg(p.part_lse + blk * kT + r) : -INFINITY;
                    const float mx = fmaxf(lse_own, lse_tail);
                    float w_own = 0.f, w_tail = 0.f, lse_n = -INFINITY;
                    if (mx > -INFINITY) {
                        const float e0 = ex2_approx((lse_own - mx) * kLog2e);
                        const float e1 = ex2_approx((lse_tail - mx) * kLog2e);
                        const float den = e0 + e1;
                        w_own = use_o ? e0 / den / l : 0.f;  // applied to the unnormalised O
                        w_tail = e1 / den;
                        lse_n = mx + lg2_approx(den) * kLn2;
                    }
                    uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(o_tm + c * 32, o);  // warp-collective: every lane loads
                        tmem_wait_ld();
                        reg_fence(o);
                        float4 tv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            tv[e] = have ? __ldcg(pblk + (c * 8 + e) * kT)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                        if (row_ok) {
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float4 x = tv[2 * e], y = tv[2 * e + 1];
                                const float* oo = reinterpret_cast<const float*>(&o[8 * e]);
                                orow[c * 4 + e] = make_uint4(
                                    pack_bf16x2(fmaf(w_own, oo[0], w_tail * x.x),
                                                fmaf(w_own, oo[1], w_tail * x.y)),
                                    pack_bf16x2(fmaf(w_own, oo[2], w_tail * x.z),
                                                fmaf(w_own, oo[3], w_tail * x.w)),
                                    pack_bf16x2(fmaf(w_own, oo[4], w_tail * y.x),
                                                fmaf(w_own, oo[5], w_tail * y.y)),
                                    pack_bf16x2(fmaf(w_own, oo[6], w_tail * y.z),
                                                fmaf(w_own, oo[7], w_tail * y.w)));
                            }
                        }
                    }
                    if (row_ok && p.lse) p.lse[row] = lse_n;
                }
            } else if (valid) {
                const int64_t row = (int64_t)(it.b * G.Hq + hq) * p.S + (int64_t)it.i * p.Sb +
                                    (int64_t)qt * kT + r;
                // a shard's last tile may hold fewer than 128 real rows
                const bool row_ok = !RAGGED || qt < G.rg.nt - 1 || r < p.rem;
                const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
                const uint64_t inv2 = f2_pack(inv_l, inv_l);
                uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(o_tm + c * 32, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    uint32_t pkd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float lo, hi;
                        f2_unpack(f2_mul(f2_pack_u(o[e], o[e + 1]), inv2), lo, hi);
                        pkd[e / 2] = pack_bf16x2(lo, hi);
                    }
                    if (row_ok) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            orow[c * 4 + e] = make_uint4(pkd[4 * e], pkd[4 * e + 1], pkd[4 * e + 2],
                                                         pkd[4 * e + 3]);
                    }
                }
                if (p.lse && row_ok)
                    p.lse[row] = (l > 0.f) ? (m_used * sl2 + lg2_approx(l)) * 0.69314718055994531f
                                           : -INFINITY;
                if (LOG && r == 0) {
                    const int64_t unit =
                        ((int64_t)(it.b * G.Hq + hq) * G.rg.N + it.i) * G.rg.nt + qt;
                    p.counts[unit] = n_logged;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::bOEmpty + t));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
// Stream-K applies to non-causal problems with fewer than two items per SM
// (the dynamic queue's last wave would leave SMs idle) and at least one item
// per SM (so an item is cut between at most two CTAs, into a head and a
// tail).  Every item then folds the same N * nt key tiles.
static bool use_streamk(long long n_items, const FwdProblem& pr, int nt, int sm_count) {
    const long long fold_len = (long long)pr.N * nt;
    return !pr.causal && sm_count > 0 && n_items >= sm_count && n_items < 2ll * sm_count &&
           fold_len <= 0xffff && n_items < (1ll << 31);
}

// L2 size of the current device, read once per device (0 if unknown).
static long long device_l2_bytes() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0) v = -1;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v > 0 ? v : 0;
}

// The stream-K scratch (the tails' partials and flags) comes from a memory
// pool the library owns per device, allocated and freed on the launch's
// stream, so launches on different streams never share it; freed blocks stay
// reserved in the pool (up to 1 GiB) for the next launch.  Under CUDA-graph
// stream capture it is a graph allocation of the device's default pool.
static std::mutex g_pool_mu;
static cudaMemPool_t g_pool[64];

static int scratch_alloc(void** ptr, int64_t bytes, cudaStream_t stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return RA_ERR_CUDA;
    if (cap == cudaStreamCaptureStatusActive)
        return cudaMallocAsync(ptr, bytes, stream) == cudaSuccess ? RA_OK : RA_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return RA_ERR_UNSUPPORTED;
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        if (!g_pool[dev]) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t created = nullptr;
            if (cudaMemPoolCreate(&created, &props) != cudaSuccess) return RA_ERR_CUDA;
            uint64_t keep = 1ull << 30;
            if (cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep) !=
                cudaSuccess)
                return RA_ERR_CUDA;
            g_pool[dev] = created;
        }
        pool = g_pool[dev];
    }
    return cudaMallocFromPoolAsync(ptr, bytes, pool, stream) == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

template <int D, bool RAGGED>
static int launch_streamk(Params P, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, int sm_count, cudaStream_t stream, int N) {
    using C = Cfg<D>;
    P.fold_len = N * P.G.rg.nt;
    P.n_work = P.G.n_items << 32;
    const int64_t rows = P.G.n_items * 2 * kT;  // [item][slot][row]
    const int64_t o_bytes = rows * D * 4, l_bytes = (rows * 4 + 255) / 256 * 256;
    const int64_t f_bytes = P.G.n_items * 8 * 4;
    void* ws = nullptr;
    int rc = scratch_alloc(&ws, o_bytes + l_bytes + f_bytes, stream);
    if (rc) return rc;
    P.part_o = static_cast<float*>(ws);
    P.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + o_bytes);
    P.part_flag = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + o_bytes + l_bytes);
    auto kern = fwd_kernel<D, false, false, RAGGED, kModeStreamK>;
    if (cudaMemsetAsync(P.part_flag, 0, f_bytes, stream) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
            cudaSuccess) {
        rc = RA_ERR_CUDA;
    } else {
        // one CTA per SM, every CTA resident: a head segment's wait for the
        // next CTA's tail always ends
        kern<<<(unsigned)sm_count, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, P);
        if (cudaGetLastError() != cudaSuccess) rc = RA_ERR_CUDA;
    }
    if (cudaFreeAsync(ws, stream) != cudaSuccess) rc = RA_ERR_CUDA;
    return rc;
}

template <int D, bool LOG, bool RAGGED>
static int launch_impl(const FwdProblem& pr, const FoldLog* flog, unsigned int* status,
                       unsigned int* work, int sm_count, cudaStream_t stream,
                       long long timeout_cycles, int withhold_first_k, int split_mode) {
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const int64_t q_rows = (int64_t)pr.B * pr.Hq * pr.S, kv_rows = (int64_t)pr.B * pr.Hkv * pr.S;
    if (!encode_rows_bf16(&mq, pr.q, q_rows, D) || !encode_rows_bf16(&mk, pr.k, kv_rows, D) ||
        !encode_rows_bf16(&mv, pr.v, kv_rows, D))
        return RA_ERR_CUDA;
    Params P = {};
    const int Sb = (int)(pr.S / pr.N);
    const int nt = (Sb + kT - 1) / kT;
    P.G = make_item_geom(pr.B, pr.Hq, pr.Hkv, pr.N, nt, pr.causal, pr.striped);
    P.S = pr.S;
    P.Sb = Sb;
    P.rem = Sb - (nt - 1) * kT;
    P.sl2 = (float)((double)pr.scale * 1.4426950408889634);
    P.out = static_cast<__nv_bfloat16*>(pr.out);
    P.lse = pr.lse;
    P.status = status;
    P.log = flog ? flog->log : nullptr;
    P.counts = flog ? flog->counts : nullptr;
    P.max_entries = flog ? flog->max_entries : 0;
    P.work = work;
    P.timeout_cycles = timeout_cycles > 0 ? timeout_cycles : kTimeoutCycles;
    P.n_work = P.G.n_items;
    if (P.G.n_items <= 0) return RA_OK;
    if (!LOG && !withhold_first_k && split_mode == 1 && use_streamk(P.G.n_items, pr, nt, sm_count))
        return launch_streamk<D, RAGGED>(P, mq, mk, mv, sm_count, stream, pr.N);
    if (cudaMemsetAsync(work, 0, sizeof(unsigned int), stream) != cudaSuccess) return RA_ERR_CUDA;
    auto kern = withhold_first_k ? fwd_kernel<D, false, true, RAGGED>
                                 : fwd_kernel<D, LOG, false, RAGGED>;
    const long long grid = P.G.n_items < sm_count ? P.G.n_items : sm_count;
    // large blocks: every query shard enters the ring at block N-1 (the
    // logging and self-test variants keep the ring order)
    if (!LOG && !withhold_first_k && ring_entry(P.G, grid, Sb, D, device_l2_bytes()))
        kern = fwd_kernel<D, false, false, RAGGED, kModeRingFromLast>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return RA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

template <int D, bool RAGGED>
static int launch_step_impl(const StepProblem& pr, unsigned int* status, unsigned int* work,
                            int sm_count, cudaStream_t stream) {
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const int64_t q_rows = (int64_t)pr.B * pr.Hq * pr.Sb, kv_rows = (int64_t)pr.B * pr.Hkv * pr.Sb;
    if (!encode_rows_bf16(&mq, pr.q, q_rows, D) || !encode_rows_bf16(&mk, pr.k, kv_rows, D) ||
        !encode_rows_bf16(&mv, pr.v, kv_rows, D))
        return RA_ERR_CUDA;
    Params P = {};
    const int Sb = (int)pr.Sb;
    const int nt = (Sb + kT - 1) / kT;
    // items: the query tiles of the one local shard (a ring of one device);
    // the masks come from the real ring
    P.G = make_item_geom(pr.B, pr.Hq, pr.Hkv, 1, nt, pr.causal, pr.layout);
    P.ring = RingGeom{pr.N, nt, pr.causal, pr.layout};
    P.step_i = pr.i;
    P.step_j = pr.j;
    P.step_s = ((pr.i - pr.j) % pr.N + pr.N) % pr.N;
    P.step_first = pr.first;
    P.step_last = pr.last;
    P.state_o = pr.state_o;
    P.state_lse = pr.state_lse;
    P.S = Sb;
    P.Sb = Sb;
    P.rem = Sb - (nt - 1) * kT;
    P.sl2 = (float)((double)pr.scale * 1.4426950408889634);
    P.out = static_cast<__nv_bfloat16*>(pr.out);
    P.lse = pr.lse;
    P.status = status;
    P.work = work;
    P.timeout_cycles = kTimeoutCycles;
    P.n_work = P.G.n_items;
    if (P.G.n_items <= 0) return RA_OK;
    if (cudaMemsetAsync(work, 0, sizeof(unsigned int), stream) != cudaSuccess) return RA_ERR_CUDA;
    auto kern = fwd_kernel<D, false, false, RAGGED, kModeStep>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return RA_ERR_CUDA;
    const long long grid = P.G.n_items < sm_count ? P.G.n_items : sm_count;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

}  // namespace tc

bool tc_step_supported(const StepProblem& p) {
    if (p.D != 64 && p.D != 128) return false;
    if (p.Sb <= 0 || p.Sb > (1ll << 30)) return false;
    if (p.layout == kZigzag && p.Sb % (2 * tc::kT)) return false;
    if ((int64_t)p.B * p.Hq * p.Sb >= (1ll << 31) || (int64_t)p.B * p.Hkv * p.Sb >= (1ll << 31))
        return false;
    return true;
}

int launch_tc_step(const StepProblem& p, unsigned int* status, unsigned int* work, int sm_count,
                   cudaStream_t stream) {
    if (!tc_step_supported(p)) return RA_ERR_UNSUPPORTED;
    if (!work) return RA_ERR_INVALID_ARG;
    const bool ragged = p.Sb % tc::kT != 0;
    if (p.D == 128)
        return ragged ? tc::launch_step_impl<128, true>(p, status, work, sm_count, stream)
                      : tc::launch_step_impl<128, false>(p, status, work, sm_count, stream);
    return ragged ? tc::launch_step_impl<64, true>(p, status, work, sm_count, stream)
                  : tc::launch_step_impl<64, false>(p, status, work, sm_count, stream);
}

bool tc_supported(const FwdProblem& p) {
    if (p.dtype != RA_BF16 || (p.D != 64 && p.D != 128)) return false;
    if (p.S % p.N) return false;
    const int64_t Sb = p.S / p.N;
    // a ragged last tile per shard is supported for contiguous and striped
    // shards; zigzag chunks must be whole tiles
    if (p.striped == kZigzag && Sb % (2 * tc::kT)) return false;
    if (Sb > (1ll << 30)) return false;
    if ((int64_t)p.B * p.Hq * p.S >= (1ll << 31) || (int64_t)p.B * p.Hkv * p.S >= (1ll << 31))
        return false;
    return true;
}

bool tc_uses_streamk(const FwdProblem& p, int sm_count) {
    if (!tc_supported(p)) return false;
    const int Sb = (int)(p.S / p.N);
    const int nt = (Sb + tc::kT - 1) / tc::kT;
    const ItemGeom G = make_item_geom(p.B, p.Hq, p.Hkv, p.N, nt, p.causal, p.striped);
    return tc::use_streamk(G.n_items, p, nt, sm_count);
}

int launch_tc(const FwdProblem& p, const FoldLog* flog, unsigned int* status, unsigned int* work,
              int sm_count, cudaStream_t stream, long long timeout_cycles, int withhold_first_k,
              int split_mode) {
    if (!tc_supported(p)) return RA_ERR_UNSUPPORTED;
    if (!work) return RA_ERR_INVALID_ARG;
    const bool ragged = (p.S / p.N) % tc::kT != 0;
    auto go = [&](auto d, auto lg, auto rg) {
        return tc::launch_impl<decltype(d)::value, decltype(lg)::value, decltype(rg)::value>(
            p, flog, status, work, sm_count, stream, timeout_cycles, withhold_first_k,
            split_mode);
    };
    using T = std::true_type;
    using F = std::false_type;
    using D128 = std::integral_constant<int, 128>;
    using D64 = std::integral_constant<int, 64>;
    if (p.D == 128) {
        if (flog) return ragged ? go(D128{}, T{}, T{}) : go(D128{}, T{}, F{});
        return ragged ? go(D128{}, F{}, T{}) : go(D128{}, F{}, F{});
    }
    if (flog) return ragged ? go(D64{}, T{}, T{}) : go(D64{}, T{}, F{});
    return ragged ? go(D64{}, F{}, T{}) : go(D64{}, F{}, F{});
}

}  // namespace ra
