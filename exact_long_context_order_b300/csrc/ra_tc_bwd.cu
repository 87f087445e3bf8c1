// Tensor-core (tcgen05) ring-attention backward for sm_103a: bf16 in, fp32
// accumulate, head dimension 128.
//
// The gradients are the chain rule of the forward; the pages give training as
// the method's use (the Italian aiunderstanding.org page, "Implementazione nel
// mondo reale": 1M-token LLM training; the glossary page: end-to-end training
// throughput) without writing the backward out.  With P = exp(scale q.k - lse)
// and delta = dO.O per query row:
//   dS = P (dO.v - delta),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// The work is split between two persistent kernels so that neither needs
// atomics and the results do not depend on scheduling:
//  * dq_kernel: one 128-row query tile per work item, folding the key/value
//    tiles of the forward's fold list in ring order (dQ of shard i stays on
//    device i, like the forward's output).  Per key tile: S = Q K^T and
//    dP = dO V^T (SS MMAs into TMEM); the softmax warps form dS in registers
//    and write it (bf16) over S; dQ += dS K (A from TMEM, K read MN-major).
//  * dkv_kernel: one 128-row key tile per work item.  Its dK and dV
//    accumulators travel with the block round the ring in its cyclic order,
//    entering it at device 0 (query shards i = 0..N-1, so that blocks running
//    together read the same query tiles from L2), and in each shard the
//    query tiles that see it, for every query head of its GQA group.  Each
//    query tile is taken as two halves of 64 rows with their own TMEM
//    columns: S^T = K Q^T and dP^T = V dO^T per half; P^T and dS^T (bf16) are
//    written over them; dV += P^T dO and dK += dS^T Q (A from TMEM, dO and Q
//    read MN-major).  Each half is its own dependency chain, so the next
//    tile's half follows this tile's same half without waiting for the other.
// Both kernels recompute S and dP, so a tile pair costs 7 tile GEMMs where a
// single kernel reducing dQ across key tiles would cost 5.
//
// Both use one CTA per SM (384 threads): warp 0 lane 0 issues TMA copies,
// lane 0 of two warps issues MMAs (while one issuer waits for a softmax
// signal, the other's GEMMs keep the tensor core busy): warps 1 and 3 in
// dq_kernel, warps 1 and 2 in dkv_kernel, where warp 3 stages the per-row lse
// and delta of each query tile; warp 2 owns TMEM; warps 4-11 are two
// warpgroups that split the 128 columns of each score tile (in dkv_kernel,
// one query half each).  Every mbarrier
// wait is bounded; on time-out a kernel records kStatusTimeout, drains its
// in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "ra.h"
#include "schedule.cuh"
#include "tmap.h"
#include "waits.cuh"

namespace ra {
namespace tcb {

constexpr int kT = 128;                    // query and key tile rows
constexpr int kD = 128;                    // largest head dimension (sizes the smem slots)
constexpr int kBoxBytes = kT * 128;        // 128 rows x 64 bf16 columns (128-byte swizzle)
constexpr int kTileBytes = kT * kD * 2;    // one smem slot: two boxes
// A D = 64 tile fills the first box of its slot; D = 128 fills both.
constexpr int kThreads = 384;
constexpr long long kTimeoutCycles = 4000000000ll;
constexpr long long kDrainCycles = 400000000ll;
// 384 threads launched at 168 registers; warps 0-3 drop to 80, the two
// softmax warpgroups rise to 208: 128*80 + 256*208 = 63488 <= 64512.
constexpr uint32_t kRegsOther = 80, kRegsSoftmax = 208;
constexpr float kLog2e = 1.4426950408889634f;

// D (+)= A B^T for two K-major 128 x HD bf16 tiles in smem (HD/16 K-steps of 16).
template <int HD>
__device__ __forceinline__ void mma_nt(uint32_t d_tm, uint32_t a_smem, uint32_t b_smem,
                                       bool acc) {
    constexpr uint32_t idesc = make_idesc_bf16(128, 128, false, false);
    const uint64_t da = make_sdesc(a_smem, 16, 1024, kLayoutSW128);
    const uint64_t db = make_sdesc(b_smem, 16, 1024, kLayoutSW128);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off16 = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
        umma_ss(d_tm, da + off16, db + off16, idesc, (acc || kk > 0) ? 1u : 0u);
    }
}

// D (+)= A B: A is 128 x 128 bf16 in TMEM (two values per column), B a
// row-major 128 x HD tile in smem read MN-major (8 K-steps of 16 rows).
template <int HD>
__device__ __forceinline__ void mma_tn(uint32_t d_tm, uint32_t a_tm, uint32_t b_smem, bool acc) {
    constexpr uint32_t idesc = make_idesc_bf16(128, HD, false, true);
    const uint64_t db = make_sdesc(b_smem, kBoxBytes, 1024, kLayoutSW128);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        umma_ts(d_tm, a_tm + kk * 8, db + (uint64_t)((kk * 2048) >> 4), idesc,
                (acc || kk > 0) ? 1u : 0u);
}

// Half tiles of the dk/dv kernel: 64 of a query tile's 128 rows, starting
// 64 rows (8 KiB of 128-byte rows) into each box of the smem slot.
constexpr uint32_t kHalfBytes = 64 * 128;

// D = A B^T for a K-major 128 x HD tile A and the 64 K-major rows of B at
// b_smem (M = 128, N = 64, HD/16 K-steps of 16).
template <int HD>
__device__ __forceinline__ void mma_nt_n64(uint32_t d_tm, uint32_t a_smem, uint32_t b_smem) {
    constexpr uint32_t idesc = make_idesc_bf16(128, 64, false, false);
    const uint64_t da = make_sdesc(a_smem, 16, 1024, kLayoutSW128);
    const uint64_t db = make_sdesc(b_smem, 16, 1024, kLayoutSW128);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off16 = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
        umma_ss(d_tm, da + off16, db + off16, idesc, kk > 0 ? 1u : 0u);
    }
}

// D (+)= A B: A is 128 x 64 bf16 in TMEM (32 columns), B the 64 row-major
// rows of HD columns at b_smem, read MN-major (4 K-steps of 16 rows).
template <int HD>
__device__ __forceinline__ void mma_tn_k64(uint32_t d_tm, uint32_t a_tm, uint32_t b_smem,
                                           bool acc) {
    constexpr uint32_t idesc = make_idesc_bf16(128, HD, false, true);
    const uint64_t db = make_sdesc(b_smem, kBoxBytes, 1024, kLayoutSW128);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        umma_ts(d_tm, a_tm + kk * 8, db + (uint64_t)((kk * 2048) >> 4), idesc,
                (acc || kk > 0) ? 1u : 0u);
}

struct Params {
    TileGeom G;
    int64_t S;
    int Sb;
    int rem;      // rows of each shard's last tile
    float sl2;    // scale * log2(e)
    float scale;
    const float* lse;
    const float* delta;
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    unsigned int* status;
    unsigned int* work;
    long long timeout_cycles;  // self test only: limit of every bounded wait
    // Ring step only (STEP kernels): the buffers hold query shard step_i (q,
    // dout, lse, delta) and key/value block step_j alone, S = Sb rows per
    // (b, h) slice, so the item geometry is a ring of one device; `ring` is
    // the real ring whose masks apply.  The step adds its terms into fp32
    // state: dq_state for the shard's rows, dk_state / dv_state for the
    // block's (the accumulators that travel with the block).  step_first:
    // the state starts at zero; step_last: the totals go to dq, dk, dv in
    // bf16 instead of back to the state.
    RingGeom ring;
    int step_i, step_j, step_first, step_last;
    float* dq_state;
    float* dk_state;
    float* dv_state;
};

// The walks of the ring-step kernels (one block of the real ring).
// dq: key tiles [0, nk) of block step_j that query tile qt of shard step_i
// sees.
RA_HD void step_key_walk(const Params& p, int qt, TileWalk& w) {
    int d;
    w.s = 0;
    w.j = p.step_j;
    w.kt = 0;
    shard_span(p.ring, p.step_i, p.step_j, qt, &w.nk, &d);
}
// dk/dv: the query tiles of shard step_i (every query head of the group)
// that key tile kt of block step_j sees; w.i is 0 (the buffers' only shard)
// while the walk runs and 1 once it is done.
RA_HD void step_query_walk(const Params& p, int kt, KeyWalk& w) {
    key_span(p.ring, p.step_i, p.step_j, kt, &w.q_lo, &w.q_hi);
    w.s = 0;
    w.gi = 0;
    w.qt = w.q_lo;
    w.i = (w.q_lo < w.q_hi) ? 0 : 1;
}
RA_HD void step_query_next(KeyWalk& w, int heads) {
    if (++w.qt < w.q_hi) return;
    w.qt = w.q_lo;
    if (++w.gi < heads) return;
    w.i = 1;
}

// ============================================================== dq kernel
namespace dqk {
// K tiles are read by S(n) and, a tile later, by dQ(n): three stages keep the
// next load in flight; V tiles are read only by dP(n): two stages.
constexpr int kKStages = 3, kVStages = 2;
constexpr int kQOff = 0, kDOOff = kTileBytes, kKOff = 2 * kTileBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kBarOff = kVOff + kVStages * kTileBytes;
enum {
    bQFull = 0, bQEmpty, bKFull, bKEmpty = bKFull + kKStages, bVFull = bKEmpty + kKStages,
    bVEmpty = bVFull + kVStages, bSFull = bVEmpty + kVStages, bDPFull = bSFull + 2, bSRead,
    bDsFull, bDqFull = bDsFull + 2, bDqEmpty, bDrain, bItemFull = bDrain + 2,
    bItemEmpty = bItemFull + 2, kNumBars = bItemEmpty + 2
};
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 32 + 1024;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColDP = 256, kColDQ = 384;
constexpr uint32_t kItemReaders = 10;  // two MMA issuers and eight softmax warps
}  // namespace dqk

// SELFTEST: the failure-detection self test (the first K tile is never
// loaded, every wait is bounded by p.timeout_cycles).  STEP: one step of a
// ring whose devices are separate processes (see Params).
template <int D, bool SELFTEST, bool STEP = false, bool FROM_LAST = false>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const Params p) {
    using namespace dqk;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kBarOff + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile long long* item_slot = reinterpret_cast<volatile long long*>(tmem_slot + 2);  // [2]
    auto bar = [&](int idx) -> uint32_t { return base + kBarOff + idx * 8; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TileGeom& G = p.G;
    const int nt = G.rg.nt;
    // limits of the bounded waits (the self test uses a short one)
    const long long wlim = SELFTEST ? p.timeout_cycles : kTimeoutCycles;
    const long long dlim = SELFTEST ? p.timeout_cycles : kDrainCycles;
    constexpr int kLoadBytes = kT * D * 2;  // bytes of one q, k, v or dout tile

    if (tid == 0) {
        mbar_init(bar(bQFull), 1);
        mbar_init(bar(bQEmpty), 2);  // S reads Q (issuer A), dP reads dO (issuer B)
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(bKFull + s), 1);
            mbar_init(bar(bKEmpty + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(bVFull + s), 1);
            mbar_init(bar(bVEmpty + s), 1);
        }
        mbar_init(bar(bSFull + 0), 1);
        mbar_init(bar(bSFull + 1), 1);
        mbar_init(bar(bDPFull), 1);
        mbar_init(bar(bSRead), 8);
        mbar_init(bar(bDsFull + 0), 8);
        mbar_init(bar(bDsFull + 1), 8);
        mbar_init(bar(bDqFull), 1);
        mbar_init(bar(bDqEmpty), 8);
        mbar_init(bar(bDrain), 1);
        mbar_init(bar(bDrain + 1), 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(bItemFull + t), 1);
            mbar_init(bar(bItemEmpty + t), kItemReaders);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto read_item = [&](int k, bool& ok) -> long long {
        ok = wait_bar(bar(bItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status, wlim);
        return ok ? item_slot[k & 1] : G.n_items;
    };
    auto walk_item = [&](const QTile& t) {
        Item it;
        it.b = t.b; it.kvh = t.kvh; it.i = t.i;
        it.h[0] = it.h[1] = t.h;
        it.qt[0] = it.qt[1] = t.qt;
        it.valid1 = 0;
        return it;
    };
    // the item's key tiles: its fold list (entered at block N-1 with
    // FROM_LAST), or in a ring step block step_j's
    using Walk = typename std::conditional<FROM_LAST, TileWalkFromLast, TileWalk>::type;
    auto wstart = [&](Walk& w, const Item& it) {
        if constexpr (STEP) step_key_walk(p, it.qt[0], w);
        else w.start(G.rg, it);
    };
    auto wdone = [&](const Walk& w) -> bool {
        if constexpr (STEP) return w.kt >= w.nk;
        else return w.done(G.rg);
    };
    auto wnext = [&](Walk& w, const Item& it) {
        if constexpr (STEP) ++w.kt;
        else w.next(G.rg, it);
    };

    if (warp < 4) regs_dec<kRegsOther>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            uint32_t tiles = 0, q_loads = 0;  // key tiles loaded (K and V ring positions)
            int k = 0;
            bool ok = true;
            auto publish = [&](int kk, long long v) -> bool {
                if (kk >= 2 && !wait_bar(bar(bItemEmpty + (kk & 1)), ((kk >> 1) - 1) & 1,
                                         abort_flag, p.status, wlim))
                    return false;
                item_slot[kk & 1] = v;
                mbar_arrive(bar(bItemFull + (kk & 1)));
                return true;
            };
            long long item = (long long)atomicAdd(p.work, 1u);
            ok = publish(0, item);
            for (; ok && item < G.n_items; ++k) {
                const long long next = (long long)atomicAdd(p.work, 1u);
                if (!(ok = publish(k + 1, next))) break;
                const QTile t = decode_qtile(G, item);
                const Item it = walk_item(t);
                item = next;
                if (k > 0 && !(ok = wait_bar(bar(bQEmpty), (k - 1) & 1, abort_flag, p.status,
                                             wlim)))
                    break;
                mbar_arrive_expect_tx(bar(bQFull), 2 * kLoadBytes);
                ++q_loads;
                const int qrow = (int)((int64_t)(t.b * G.Hq + t.h) * p.S + (int64_t)t.i * p.Sb +
                                       (int64_t)t.qt * kT);
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load_2d(base + kQOff + bx * kBoxBytes, &tm_q, bx * 64, qrow, bar(bQFull),
                                pol_q);
                    tma_load_2d(base + kDOOff + bx * kBoxBytes, &tm_do, bx * 64, qrow,
                                bar(bQFull), pol_q);
                }
                const int64_t kvrow0 = (int64_t)(t.b * G.Hkv + t.kvh) * p.S;
                Walk w;
                for (wstart(w, it); !wdone(w) && ok; wnext(w, it), ++tiles) {
                    const int64_t jrow = STEP ? 0 : (int64_t)w.j * p.Sb;
                    const int row = (int)(kvrow0 + jrow + (int64_t)w.kt * kT);
                    const uint32_t sk = tiles % kKStages, uk = tiles / kKStages;
                    if (uk > 0 && !(ok = wait_bar(bar(bKEmpty + sk), (uk - 1) & 1, abort_flag,
                                                  p.status, wlim)))
                        break;
                    if (!(SELFTEST && tiles == 0)) {  // self test: K of the first tile never comes
                        mbar_arrive_expect_tx(bar(bKFull + sk), kLoadBytes);
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_load_2d(base + kKOff + sk * kTileBytes + bx * kBoxBytes, &tm_k,
                                        bx * 64, row, bar(bKFull + sk), pol_kv);
                    }
                    const uint32_t sv = tiles % kVStages, uv = tiles / kVStages;
                    if (uv > 0 && !(ok = wait_bar(bar(bVEmpty + sv), (uv - 1) & 1, abort_flag,
                                                  p.status, wlim))) {
                        ++tiles;  // K of this tile is in flight
                        break;
                    }
                    mbar_arrive_expect_tx(bar(bVFull + sv), kLoadBytes);
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_load_2d(base + kVOff + sv * kTileBytes + bx * kBoxBytes, &tm_v,
                                    bx * 64, row, bar(bVFull + sv), pol_kv);
                }
            }
            if (!ok) {
                // let every copy that may still be in flight land before exit
                if (q_loads > 0) drain_wait(bar(bQFull), (q_loads - 1) & 1, dlim);
                for (uint32_t pos = tiles > (uint32_t)kKStages ? tiles - kKStages : 0; pos < tiles;
                     ++pos)
                    drain_wait(bar(bKFull + pos % kKStages), (pos / kKStages) & 1, dlim);
                for (uint32_t pos = tiles > (uint32_t)kVStages ? tiles - kVStages : 0; pos < tiles;
                     ++pos)
                    drain_wait(bar(bVFull + pos % kVStages), (pos / kVStages) & 1, dlim);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA issuers
        // Lane 0 of warp 1 (A): S(n) into S[n&1], then dQ += dS(n-1) K(n-1) once the
        // softmax has written dS(n-1) over S[(n-1)&1].  Lane 0 of warp 3 (B):
        // dP(n) into DP once the softmax has read dP(n-1).  Two threads, so that
        // one's waits on the softmax overlap the other's GEMMs in the pipe.
        // "S ready" is doubled by tile parity: A may run a tile ahead of B.
        if (lane == 0) {
            const bool is_a = (warp == 1);
            uint32_t g = 0;  // key tiles issued so far (ring positions of K and V)
            int k = 0;
            bool ok = true;
            auto sbuf = [&](uint32_t gg) { return tmem + ((gg & 1) ? kColS1 : kColS0); };
            auto issue_dq = [&](uint32_t n, int kk) -> bool {
                // dq of tile g-1: needs its dS and, for the item's first, a drained DQ
                if (!wait_bar(bar(bDsFull + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_flag,
                              p.status, wlim))
                    return false;
                if (n == 1 && kk > 0 &&
                    !wait_bar(bar(bDqEmpty), (kk - 1) & 1, abort_flag, p.status, wlim))
                    return false;
                tc_fence_after();
                const uint32_t sk = (g - 1) % kKStages;
                mma_tn<D>(tmem + kColDQ, sbuf(g - 1), base + kKOff + sk * kTileBytes, n > 1);
                umma_commit(bar(bKEmpty + sk));
                return true;
            };
            for (;; ++k) {
                const long long item = read_item(k, ok);
                if (ok) mbar_arrive(bar(bItemEmpty + (k & 1)));
                if (!ok || item >= G.n_items) break;
                const Item it = walk_item(decode_qtile(G, item));
                if (!(ok = wait_bar(bar(bQFull), k & 1, abort_flag, p.status, wlim)))
                    break;
                Walk w;
                uint32_t n = 0;
                for (wstart(w, it); !wdone(w); wnext(w, it), ++n) {
                    if (is_a) {
                        const uint32_t sk = g % kKStages;
                        if (!(ok = wait_bar(bar(bKFull + sk), (g / kKStages) & 1, abort_flag,
                                            p.status, wlim)))
                            break;
                        tc_fence_after();
                        mma_nt<D>(sbuf(g), base + kQOff, base + kKOff + sk * kTileBytes, false);
                        umma_commit(bar(bSFull + (g & 1)));
                        if (n > 0 && !(ok = issue_dq(n, k))) break;
                    } else {
                        const uint32_t sv = g % kVStages;
                        if (!(ok = wait_bar(bar(bVFull + sv), (g / kVStages) & 1, abort_flag,
                                            p.status, wlim)))
                            break;
                        if (g > 0 && !(ok = wait_bar(bar(bSRead), (g - 1) & 1, abort_flag,
                                                     p.status, wlim)))
                            break;
                        tc_fence_after();
                        mma_nt<D>(tmem + kColDP, base + kDOOff, base + kVOff + sv * kTileBytes, false);
                        umma_commit(bar(bDPFull));
                        umma_commit(bar(bVEmpty + sv));
                    }
                    ++g;
                }
                if (!ok) break;
                umma_commit(bar(bQEmpty));  // this issuer's MMAs reading Q (A) or dO (B) are issued
                if (is_a) {
                    if (STEP && n == 0) {
                        // the block holds no key this tile sees: no dQ MMA; the
                        // epilogue folds nothing into the state
                        mbar_arrive(bar(bDqFull));
                    } else {
                        if (!(ok = issue_dq(n, k))) break;
                        umma_commit(bar(bDqFull));
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                umma_commit(bar(bDrain + (is_a ? 0 : 1)));
                drain_wait(bar(bDrain + (is_a ? 0 : 1)), 0, dlim);
            }
        }
    } else if (warp < 4) {
        // warp 2 owns TMEM
    } else {
        // ------------------------------------------------------------ softmax
        regs_inc<kRegsSoftmax>();
        const int wg = (warp - 4) >> 2;        // key columns [64 wg, 64 wg + 64)
        const int r = (warp & 3) * 32 + lane;  // query row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int c0 = 64 * wg;
        const uint64_t sl2x2 = f2_pack(p.sl2, p.sl2);
        uint32_t g = 0;
        int k = 0;
        bool ok = true;
        for (;; ++k) {
            const long long item = read_item(k, ok);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bItemEmpty + (k & 1)));
            if (item >= G.n_items) break;
            const QTile t = decode_qtile(G, item);
            const Item it = walk_item(t);
            const int64_t row = (int64_t)(t.b * G.Hq + t.h) * p.S + (int64_t)t.i * p.Sb +
                                (int64_t)t.qt * kT + r;
            const bool row_ok = t.qt < nt - 1 || r < p.rem;
            const float nl2 = row_ok ? -p.lse[row] * kLog2e : 0.f;
            const float dl = row_ok ? p.delta[row] : 0.f;
            const uint64_t nl2x2 = f2_pack(nl2, nl2), ndl2 = f2_pack(-dl, -dl);
            Walk w;
            uint32_t n = 0;
            for (wstart(w, it); !wdone(w); wnext(w, it), ++g, ++n) {
                const int kind = STEP ? fold_kind(p.ring, p.step_i, p.step_j, t.qt, w.kt)
                                      : fold_kind(G.rg, t.i, w.j, t.qt, w.kt);
                ok = wait_bar(bar(bSFull + (g & 1)), (g >> 1) & 1, abort_flag, p.status,
                              wlim) &&
                     wait_bar(bar(bDPFull), g & 1, abort_flag, p.status, wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sb = tmem + lane_off + ((g & 1) ? kColS1 : kColS0);
                uint32_t sr[2][32], dp[2][32];
                tmem_ld32(sb + c0, sr[0]);
                tmem_ld32(sb + c0 + 32, sr[1]);
                tmem_ld32(tmem + lane_off + kColDP + c0, dp[0]);
                tmem_ld32(tmem + lane_off + kColDP + c0 + 32, dp[1]);
                tmem_wait_ld();
                reg_fence(sr[0]);
                reg_fence(sr[1]);
                reg_fence(dp[0]);
                reg_fence(dp[1]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bSRead));
                // visible iff key column <= lim
                int lim = (kind == kIncl) ? r : (kind == kStrict) ? r - 1 : kT - 1;
                if (w.kt == nt - 1 && p.rem - 1 < lim) lim = p.rem - 1;
                if (!row_ok || kind == kNone) lim = -1;
                uint32_t pk[32];
                // dS for two columns c, c + 1 of pair index e of chunk cc
                auto ds2 = [&](int cc, int e, float p0, float p1) {
                    const uint64_t dd = f2_add(f2_pack_u(dp[cc][e], dp[cc][e + 1]), ndl2);
                    float d0, d1;
                    f2_unpack(f2_mul(f2_pack(p0, p1), dd), d0, d1);
                    pk[cc * 16 + e / 2] = pack_bf16x2(d0, d1);
                };
                if (lim >= kT - 1) {  // every pair of the tile is visible
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float a0, a1;
                            f2_unpack(f2_fma(f2_pack_u(sr[cc][e], sr[cc][e + 1]), sl2x2, nl2x2),
                                      a0, a1);
                            ds2(cc, e, ex2_approx(a0), ex2_approx(a1));
                        }
                } else {
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int c = c0 + cc * 32 + e;
                            float a0, a1;
                            f2_unpack(f2_fma(f2_pack_u(sr[cc][e], sr[cc][e + 1]), sl2x2, nl2x2),
                                      a0, a1);
                            ds2(cc, e, (c <= lim) ? ex2_approx(a0) : 0.f,
                                (c + 1 <= lim) ? ex2_approx(a1) : 0.f);
                        }
                }
                // both warpgroups must have read S before dS goes over it
                ok = wait_bar(bar(bSRead), g & 1, abort_flag, p.status, wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tmem_st32(sb + 32 * wg, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bDsFull + (g & 1)));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            ok = wait_bar(bar(bDqFull), k & 1, abort_flag, p.status, wlim);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const uint64_t sc2 = f2_pack(p.scale, p.scale);
            const int e0 = (D / 2) * wg;  // dq columns of this warpgroup
            uint4* drow = reinterpret_cast<uint4*>(p.dq + row * D + e0);
            if constexpr (STEP) {
                // dq_state (+)= scale * this block's dQ; the last step writes dq
                float4* srow = reinterpret_cast<float4*>(p.dq_state + row * D + e0);
#pragma unroll 1
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t o[32];
                    if (n > 0) {
                        tmem_ld32(tmem + lane_off + kColDQ + e0 + cc * 32, o);
                        tmem_wait_ld();
                        reg_fence(o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    float nv[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) nv[e] = p.scale * __uint_as_float(o[e]);
                    if (!row_ok) continue;
                    if (!p.step_first) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 sv = srow[cc * 8 + e];
                            nv[4 * e] += sv.x;
                            nv[4 * e + 1] += sv.y;
                            nv[4 * e + 2] += sv.z;
                            nv[4 * e + 3] += sv.w;
                        }
                    }
                    if (p.step_last) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            drow[cc * 4 + e] = make_uint4(
                                pack_bf16x2(nv[8 * e], nv[8 * e + 1]),
                                pack_bf16x2(nv[8 * e + 2], nv[8 * e + 3]),
                                pack_bf16x2(nv[8 * e + 4], nv[8 * e + 5]),
                                pack_bf16x2(nv[8 * e + 6], nv[8 * e + 7]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            srow[cc * 8 + e] = make_float4(nv[4 * e], nv[4 * e + 1],
                                                           nv[4 * e + 2], nv[4 * e + 3]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bDqEmpty));
                continue;
            }
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + kColDQ + e0 + cc * 32, o);
                tmem_wait_ld();
                reg_fence(o);
                uint32_t pkd[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float lo, hi;
                    f2_unpack(f2_mul(f2_pack_u(o[e], o[e + 1]), sc2), lo, hi);
                    pkd[e / 2] = pack_bf16x2(lo, hi);
                }
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        drow[cc * 4 + e] =
                            make_uint4(pkd[4 * e], pkd[4 * e + 1], pkd[4 * e + 2], pkd[4 * e + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bDqEmpty));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================== dk/dv kernel
namespace dkv {
constexpr int kQStages = 2, kDOStages = 2;
constexpr int kKOff = 0, kVOff = kTileBytes, kQOff = 2 * kTileBytes;
constexpr int kDOOff = kQOff + kQStages * kTileBytes;
constexpr int kVecOff = kDOOff + kDOStages * kTileBytes;  // per stage: -lse*log2e[128], delta[128]
constexpr int kVecBytes = 2 * kT * 4;
constexpr int kBarOff = kVecOff + 2 * kVecBytes;
enum {
    // a query tile's Q and dO land in the same stage and complete on one barrier,
    // so each issuer's wait for its score GEMM's input also covers the input of
    // its accumulation GEMM (the other of the two)
    bKVFull = 0, bKVEmpty, bQDFull, bQDEmpty = bQDFull + kQStages,
    bVecFull = bQDEmpty + kQStages, bVecEmpty = bVecFull + 2,
    // per query half h of the tile: S^T(h) done, P^T(h) written, dP^T(h) done, dS^T(h) written
    bSFull = bVecEmpty + 2, bPFull = bSFull + 2, bDPFull = bPFull + 2, bDsFull = bDPFull + 2,
    bAccFull = bDsFull + 2, bAccEmpty,
    bDrain, bItemFull = bDrain + 2, bItemEmpty = bItemFull + 2, kNumBars = bItemEmpty + 2
};
constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 32 + 1024;
// S^T of query half h in columns [64h, 64h + 64) (P^T written over the first
// 32 of them), dP^T of half h at 128 + 64h (dS^T over its first 32), then dV, dK.
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;
// readers of a published item: two MMA issuers, the row-vector warp, eight softmax warps
constexpr uint32_t kItemReaders = 11;
}  // namespace dkv

// SELFTEST: the failure-detection self test (the first Q tile is never
// loaded, every wait is bounded by p.timeout_cycles).  STEP: one step of a
// ring whose devices are separate processes (see Params).
template <int D, bool SELFTEST, bool STEP = false>
__global__ void __launch_bounds__(kThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const Params p) {
    using namespace dkv;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    float* vec = reinterpret_cast<float*>(gbase + kVecOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kBarOff + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile long long* item_slot = reinterpret_cast<volatile long long*>(tmem_slot + 2);  // [2]
    auto bar = [&](int idx) -> uint32_t { return base + kBarOff + idx * 8; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TileGeom& G = p.G;
    const int nt = G.rg.nt, heads = G.g;
    // limits of the bounded waits (the self test uses a short one)
    const long long wlim = SELFTEST ? p.timeout_cycles : kTimeoutCycles;
    const long long dlim = SELFTEST ? p.timeout_cycles : kDrainCycles;
    constexpr int kLoadBytes = kT * D * 2;  // bytes of one q, k, v or dout tile

    if (tid == 0) {
        // stages and accumulators used by both MMA issuers complete on two commits
        mbar_init(bar(bKVFull), 1);
        mbar_init(bar(bKVEmpty), 2);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(bQDFull + s), 1);
            mbar_init(bar(bQDEmpty + s), 2);
            mbar_init(bar(bVecFull + s), 32);
            mbar_init(bar(bVecEmpty + s), 8);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar(bSFull + h), 1);
            mbar_init(bar(bPFull + h), 4);  // the four warps of half h's warpgroup
            mbar_init(bar(bDPFull + h), 1);
            mbar_init(bar(bDsFull + h), 4);
        }
        mbar_init(bar(bAccFull), 2);
        mbar_init(bar(bAccEmpty), 8);
        mbar_init(bar(bDrain), 1);
        mbar_init(bar(bDrain + 1), 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(bItemFull + t), 1);
            mbar_init(bar(bItemEmpty + t), kItemReaders);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto read_item = [&](int k, bool& ok) -> long long {
        ok = wait_bar(bar(bItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status, wlim);
        return ok ? item_slot[k & 1] : G.n_items;
    };
    // first row of query tile (head kvh*g + gi, shard i, tile qt)
    auto qrow0 = [&](const KTile& t, const KeyWalk& w) -> int64_t {
        return (int64_t)(t.b * G.Hq + t.kvh * heads + w.gi) * p.S + (int64_t)w.i * p.Sb +
               (int64_t)w.qt * kT;
    };
    // the key tile's query tiles: in the whole ring, or in a ring step shard
    // step_i's
    auto wstart = [&](KeyWalk& w, const KTile& t) {
        if constexpr (STEP) step_query_walk(p, t.kt, w);
        else w.start(G.rg, t.j, t.kt, heads);
    };
    auto wnext = [&](KeyWalk& w, const KTile& t) {
        if constexpr (STEP) step_query_next(w, heads);
        else w.next(G.rg, t.j, t.kt, heads);
    };

    if (warp < 4) regs_dec<kRegsOther>();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_last();
            const uint64_t pol_kv = policy_evict_first();
            uint32_t g = 0, kv_loads = 0;
            int k = 0;
            bool ok = true;
            auto publish = [&](int kk, long long v) -> bool {
                if (kk >= 2 && !wait_bar(bar(bItemEmpty + (kk & 1)), ((kk >> 1) - 1) & 1,
                                         abort_flag, p.status, wlim))
                    return false;
                item_slot[kk & 1] = v;
                mbar_arrive(bar(bItemFull + (kk & 1)));
                return true;
            };
            // Q and dO of one query tile into stage g & 1, on one barrier
            auto load_stage = [&](int row) -> bool {
                const uint32_t st = g & 1, use = g >> 1;
                if (use > 0 && !wait_bar(bar(bQDEmpty + st), (use - 1) & 1, abort_flag,
                                         p.status, wlim))
                    return false;
                if (SELFTEST && g == 0) return true;  // Q(0) and dO(0) never come
                mbar_arrive_expect_tx(bar(bQDFull + st), 2 * kLoadBytes);
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load_2d(base + kQOff + st * kTileBytes + bx * kBoxBytes, &tm_q, bx * 64,
                                row, bar(bQDFull + st), pol_q);
                    tma_load_2d(base + kDOOff + st * kTileBytes + bx * kBoxBytes, &tm_do,
                                bx * 64, row, bar(bQDFull + st), pol_q);
                }
                return true;
            };
            uint32_t qd_issued = 0;
            long long item = (long long)atomicAdd(p.work, 1u);
            ok = publish(0, item);
            for (; ok && item < G.n_items; ++k) {
                const long long next = (long long)atomicAdd(p.work, 1u);
                if (!(ok = publish(k + 1, next))) break;
                const KTile t = decode_ktile(G, item);
                item = next;
                if (k > 0 && !(ok = wait_bar(bar(bKVEmpty), (k - 1) & 1, abort_flag, p.status,
                                             wlim)))
                    break;
                mbar_arrive_expect_tx(bar(bKVFull), 2 * kLoadBytes);
                ++kv_loads;
                const int krow = (int)((int64_t)(t.b * G.Hkv + t.kvh) * p.S +
                                       (int64_t)t.j * p.Sb + (int64_t)t.kt * kT);
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load_2d(base + kKOff + bx * kBoxBytes, &tm_k, bx * 64, krow, bar(bKVFull),
                                pol_kv);
                    tma_load_2d(base + kVOff + bx * kBoxBytes, &tm_v, bx * 64, krow, bar(bKVFull),
                                pol_kv);
                }
                KeyWalk w;
                for (wstart(w, t); !w.done(G.rg); wnext(w, t), ++g) {
                    if (!(ok = load_stage((int)qrow0(t, w)))) break;
                    qd_issued = g + 1;
                }
            }
            if (!ok) {
                // let every copy that may still be in flight land before exit
                if (kv_loads > 0) drain_wait(bar(bKVFull), (kv_loads - 1) & 1, dlim);
                for (uint32_t x = qd_issued > 2 ? qd_issued - 2 : 0; x < qd_issued; ++x)
                    drain_wait(bar(bQDFull + (x & 1)), (x >> 1) & 1, dlim);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA issuers
        // Two issuer threads on disjoint tensor memory, so that one's waits on
        // the softmax overlap the other's GEMMs in the pipe:
        //   lane 0 of warp 1: S^T(n, h) = K Q(n, h)^T for the two query halves h
        //   of tile n, then dV += P^T(n, h) dO(n, h) reading S^T's columns;
        //   lane 0 of warp 2: dP^T(n, h) = V dO(n, h)^T, then dK += dS^T(n, h)
        //   Q(n, h) reading dP^T's columns.
        // Each half has its own columns and its own softmax warpgroup, so the
        // next tile's S^T(n+1, h) is issued right behind dV(n, h) (in-order
        // pipe) without waiting for the other half's softmax.  Stages and
        // accumulators read by both issuers complete on two commits.
        if (lane == 0) {
            const bool is_s = (warp == 1);
            const uint32_t sc_col = tmem + (is_s ? kColS : kColDP);
            const uint32_t acc_col = tmem + (is_s ? kColDV : kColDK);
            const uint32_t a_kv = base + (is_s ? kKOff : kVOff);
            const uint32_t off_in = is_s ? kQOff : kDOOff;    // B of the score GEMM
            const uint32_t off_acc = is_s ? kDOOff : kQOff;   // B of the accumulation GEMM
            const int sig_full = is_s ? bSFull : bDPFull;
            const int sig_ready = is_s ? bPFull : bDsFull;
            uint32_t g = 0;
            int k = 0;
            bool ok = true;
            auto wait_in = [&](uint32_t gg) -> bool {
                if (!wait_bar(bar(bQDFull + (gg & 1)), (gg >> 1) & 1, abort_flag, p.status, wlim))
                    return false;
                tc_fence_after();
                return true;
            };
            // S^T(gg, h) = K Q(gg, h)^T resp. dP^T(gg, h) = V dO(gg, h)^T
            auto issue_score = [&](uint32_t gg, int h) {
                mma_nt_n64<D>(sc_col + 64 * h, a_kv,
                              base + off_in + (gg & 1) * kTileBytes + h * kHalfBytes);
                umma_commit(bar(sig_full + h));
            };
            for (;; ++k) {
                const long long item = read_item(k, ok);
                if (ok) mbar_arrive(bar(bItemEmpty + (k & 1)));
                if (!ok || item >= G.n_items) break;
                const KTile t = decode_ktile(G, item);
                if (!(ok = wait_bar(bar(bKVFull), k & 1, abort_flag, p.status, wlim)))
                    break;
                KeyWalk w;
                wstart(w, t);
                if (STEP && w.done(G.rg)) {
                    // no query tile of the shard sees this key tile: no MMA; the
                    // epilogue passes the state on unchanged
                    mbar_arrive(bar(bKVEmpty));
                    mbar_arrive(bar(bAccFull));
                    continue;
                }
                if (!(ok = wait_in(g))) break;
                issue_score(g, 0);
                issue_score(g, 1);
                for (uint32_t n = 0; !w.done(G.rg); ++n, ++g) {
                    KeyWalk nx = w;
                    wnext(nx, t);
                    const bool more = !nx.done(G.rg);
                    for (int h = 0; h < 2 && ok; ++h) {
                        // P^T(n, h) resp. dS^T(n, h) written by half h's warpgroup
                        if (!(ok = wait_bar(bar(sig_ready + h), g & 1, abort_flag, p.status,
                                            wlim)))
                            break;
                        if (n == 0 && h == 0 && k > 0 &&
                            !(ok = wait_bar(bar(bAccEmpty), (k - 1) & 1, abort_flag, p.status,
                                            wlim)))
                            break;
                        tc_fence_after();
                        mma_tn_k64<D>(acc_col, sc_col + 64 * h,
                                      base + off_acc + (g & 1) * kTileBytes + h * kHalfBytes,
                                      n > 0 || h > 0);
                        if (h == 1)  // every MMA of this tile reading Q(n) and dO(n) is issued
                            umma_commit(bar(bQDEmpty + (g & 1)));
                        if (more) {
                            if (h == 0 && !(ok = wait_in(g + 1))) break;
                            issue_score(g + 1, h);
                        }
                    }
                    if (!ok) break;
                    w = nx;
                }
                if (!ok) break;
                umma_commit(bar(bKVEmpty));
                umma_commit(bar(bAccFull));
            }
            if (!ok) {
                *abort_flag = 1;
                umma_commit(bar(bDrain + (is_s ? 0 : 1)));
                drain_wait(bar(bDrain + (is_s ? 0 : 1)), 0, dlim);
            }
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ row vectors
        // -lse * log2(e) and delta of the 128 query rows of each tile, into a
        // two-stage ring that the softmax warps read.
        uint32_t g = 0;
        int k = 0;
        bool ok = true;
        for (;; ++k) {
            const long long item = read_item(k, ok);
            if (!__all_sync(0xffffffffu, ok)) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bItemEmpty + (k & 1)));
            if (item >= G.n_items) break;
            const KTile t = decode_ktile(G, item);
            KeyWalk w;
            for (wstart(w, t); !w.done(G.rg); wnext(w, t), ++g) {
                const uint32_t st = g & 1, use = g >> 1;
                ok = use == 0 || wait_bar(bar(bVecEmpty + st), (use - 1) & 1, abort_flag, p.status,
                                          wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const int64_t row0 = qrow0(t, w);
                float* vs = vec + st * (2 * kT);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int l = lane + 32 * m;
                    const bool valid = w.qt < nt - 1 || l < p.rem;
                    vs[l] = valid ? -p.lse[row0 + l] * kLog2e : 0.f;
                    vs[kT + l] = valid ? p.delta[row0 + l] : 0.f;
                }
                mbar_arrive(bar(bVecFull + st));
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ softmax
        regs_inc<kRegsSoftmax>();
        const int wg = (warp - 4) >> 2;        // query columns [64 wg, 64 wg + 64)
        const int c = (warp & 3) * 32 + lane;  // key row of the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int q0 = 64 * wg;
        const uint64_t sl2x2 = f2_pack(p.sl2, p.sl2);
        uint32_t g = 0;
        int k = 0;
        bool ok = true;
        for (;; ++k) {
            const long long item = read_item(k, ok);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bItemEmpty + (k & 1)));
            if (item >= G.n_items) break;
            const KTile t = decode_ktile(G, item);
            const bool key_ok = t.kt < nt - 1 || c < p.rem;
            KeyWalk w;
            uint32_t n_tiles = 0;
            for (wstart(w, t); !w.done(G.rg); wnext(w, t), ++g, ++n_tiles) {
                const int kind = STEP ? fold_kind(p.ring, p.step_i, p.step_j, w.qt, t.kt)
                                      : fold_kind(G.rg, w.i, t.j, w.qt, t.kt);
                // pair (query column q, key row c) visible iff lo <= q < hi
                int lo = (kind == kIncl) ? c : (kind == kStrict) ? c + 1 : 0;
                const int hi = (w.qt == nt - 1) ? p.rem : kT;
                if (!key_ok || kind == kNone) lo = kT;
                const float* vs = vec + (g & 1) * (2 * kT);
                // ---- P^T = exp2(S^T scale log2e - lse log2e), over S^T
                ok = wait_bar(bar(bSFull + wg), g & 1, abort_flag, p.status, wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(tmem + lane_off + kColS + q0, sr[0]);
                tmem_ld32(tmem + lane_off + kColS + q0 + 32, sr[1]);
                tmem_wait_ld();
                reg_fence(sr[0]);
                reg_fence(sr[1]);
                ok = wait_bar(bar(bVecFull + (g & 1)), (g >> 1) & 1, abort_flag, p.status,
                              wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                float pf[2][32];
                uint32_t pk[32];
                const float4* nl4 = reinterpret_cast<const float4*>(vs + q0);
                // x = S^T scale log2e - lse log2e for four columns
                auto exps = [&](int cc, int e, float* x) {
                    const float4 nl = nl4[(cc * 32 + e) / 4];
                    f2_unpack(f2_fma(f2_pack_u(sr[cc][e], sr[cc][e + 1]), sl2x2,
                                     f2_pack(nl.x, nl.y)),
                              x[0], x[1]);
                    f2_unpack(f2_fma(f2_pack_u(sr[cc][e + 2], sr[cc][e + 3]), sl2x2,
                                     f2_pack(nl.z, nl.w)),
                              x[2], x[3]);
                };
                if (lo == 0 && hi == kT) {  // every pair of the tile is visible
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            float x[4];
                            exps(cc, e, x);
#pragma unroll
                            for (int m = 0; m < 4; ++m) pf[cc][e + m] = ex2_approx(x[m]);
                            pk[cc * 16 + e / 2] = pack_bf16x2(pf[cc][e], pf[cc][e + 1]);
                            pk[cc * 16 + e / 2 + 1] = pack_bf16x2(pf[cc][e + 2], pf[cc][e + 3]);
                        }
                } else {
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            float x[4];
                            exps(cc, e, x);
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const int q = q0 + cc * 32 + e + m;
                                pf[cc][e + m] = (q >= lo && q < hi) ? ex2_approx(x[m]) : 0.f;
                            }
                            pk[cc * 16 + e / 2] = pack_bf16x2(pf[cc][e], pf[cc][e + 1]);
                            pk[cc * 16 + e / 2 + 1] = pack_bf16x2(pf[cc][e + 2], pf[cc][e + 3]);
                        }
                }
                // this warpgroup alone reads and writes its half's columns
                tmem_st32(tmem + lane_off + kColS + q0, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bPFull + wg));
                // ---- dS^T = P^T (dP^T - delta), over dP^T
                ok = wait_bar(bar(bDPFull + wg), g & 1, abort_flag, p.status, wlim);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t dp[2][32];
                tmem_ld32(tmem + lane_off + kColDP + q0, dp[0]);
                tmem_ld32(tmem + lane_off + kColDP + q0 + 32, dp[1]);
                tmem_wait_ld();
                reg_fence(dp[0]);
                reg_fence(dp[1]);
                const float4* dl4 = reinterpret_cast<const float4*>(vs + kT + q0);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 dl = dl4[(cc * 32 + e) / 4];
                        float d[4];
                        f2_unpack(f2_mul(f2_pack(pf[cc][e], pf[cc][e + 1]),
                                         f2_add(f2_pack_u(dp[cc][e], dp[cc][e + 1]),
                                                f2_pack(-dl.x, -dl.y))),
                                  d[0], d[1]);
                        f2_unpack(f2_mul(f2_pack(pf[cc][e + 2], pf[cc][e + 3]),
                                         f2_add(f2_pack_u(dp[cc][e + 2], dp[cc][e + 3]),
                                                f2_pack(-dl.z, -dl.w))),
                                  d[2], d[3]);
                        pk[cc * 16 + e / 2] = pack_bf16x2(d[0], d[1]);
                        pk[cc * 16 + e / 2 + 1] = pack_bf16x2(d[2], d[3]);
                    }
                }
                tmem_st32(tmem + lane_off + kColDP + q0, pk);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(bDsFull + wg));
                    mbar_arrive(bar(bVecEmpty + (g & 1)));
                }
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            ok = wait_bar(bar(bAccFull), k & 1, abort_flag, p.status, wlim);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int64_t krow = (int64_t)(t.b * G.Hkv + t.kvh) * p.S + (int64_t)t.j * p.Sb +
                                 (int64_t)t.kt * kT + c;
            const uint64_t sc2 = f2_pack(p.scale, p.scale), one2 = f2_pack(1.f, 1.f);
            if constexpr (STEP) {
                // the block's accumulators (+)= this step's dV and scale * dK; the
                // last step writes dk, dv
#pragma unroll 1
                for (int which = 0; which < 2; ++which) {
                    const uint32_t col = which ? kColDK : kColDV;
                    const float mul = which ? p.scale : 1.f;
                    const int e0 = (D / 2) * wg;
                    float4* srow = reinterpret_cast<float4*>((which ? p.dk_state : p.dv_state) +
                                                             krow * D + e0);
                    uint4* drow = reinterpret_cast<uint4*>((which ? p.dk : p.dv) + krow * D + e0);
#pragma unroll 1
                    for (int cc = 0; cc < D / 64; ++cc) {
                        uint32_t o[32];
                        if (n_tiles > 0) {
                            tmem_ld32(tmem + lane_off + col + e0 + cc * 32, o);
                            tmem_wait_ld();
                            reg_fence(o);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = 0u;
                        }
                        if (!key_ok) continue;
                        float nv[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) nv[e] = mul * __uint_as_float(o[e]);
                        if (!p.step_first) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 sv = srow[cc * 8 + e];
                                nv[4 * e] += sv.x;
                                nv[4 * e + 1] += sv.y;
                                nv[4 * e + 2] += sv.z;
                                nv[4 * e + 3] += sv.w;
                            }
                        }
                        if (p.step_last) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                drow[cc * 4 + e] = make_uint4(
                                    pack_bf16x2(nv[8 * e], nv[8 * e + 1]),
                                    pack_bf16x2(nv[8 * e + 2], nv[8 * e + 3]),
                                    pack_bf16x2(nv[8 * e + 4], nv[8 * e + 5]),
                                    pack_bf16x2(nv[8 * e + 6], nv[8 * e + 7]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                srow[cc * 8 + e] = make_float4(nv[4 * e], nv[4 * e + 1],
                                                               nv[4 * e + 2], nv[4 * e + 3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bAccEmpty));
                continue;
            }
#pragma unroll
            for (int which = 0; which < 2; ++which) {  // dV, then dK (times scale)
                const uint32_t col = which ? kColDK : kColDV;
                const uint64_t mul = which ? sc2 : one2;
                const int e0 = (D / 2) * wg;  // dk/dv columns of this warpgroup
                uint4* drow = reinterpret_cast<uint4*>((which ? p.dk : p.dv) + krow * D + e0);
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + col + e0 + cc * 32, o);
                    tmem_wait_ld();
                    reg_fence(o);
                    uint32_t pkd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float lo2, hi2;
                        f2_unpack(f2_mul(f2_pack_u(o[e], o[e + 1]), mul), lo2, hi2);
                        pkd[e / 2] = pack_bf16x2(lo2, hi2);
                    }
                    if (key_ok) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            drow[cc * 4 + e] = make_uint4(pkd[4 * e], pkd[4 * e + 1],
                                                          pkd[4 * e + 2], pkd[4 * e + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bAccEmpty));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side
// Whether the dq kernel's query tiles enter the ring at block N-1.  Its items
// are query tiles of one head, g per (shard, tile), so the grid holds about
// grid / g query shards at once; in ring order these read as many different
// key/value blocks (4 * Sb * D bytes each per KV head).  When those exceed the
// L2, every query tile walks blocks N-1, ..., 0 instead (TileWalkFromLast), as
// the forward does, and the grid reads one block at a time.  Contiguous
// causal shards keep their global-tile order, which already shares blocks.
static bool dq_from_last(const TileGeom& G, long long grid, int Sb, int D, long long l2_bytes) {
    if ((G.rg.causal && G.rg.striped == kContiguous) || G.rg.N <= 1 || l2_bytes <= 0)
        return false;
    long long shards = (grid + G.g - 1) / G.g;
    if (shards > G.rg.N) shards = G.rg.N;
    return (double)shards * 4.0 * Sb * D > (double)l2_bytes;
}

// L2 size of the current device, read once per device (0 if unknown).
static long long l2_bytes_of_device() {
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

// kernel 0: dq_kernel over query tiles; kernel 1: dkv_kernel over key tiles
static int launch_one(const BwdProblem& pr, int which, unsigned int* status, unsigned int* work,
                      int sm_count, cudaStream_t stream, long long timeout_cycles = 0) {
    CUtensorMap mq, mdo, mk, mv;
    const int64_t q_rows = (int64_t)pr.B * pr.Hq * pr.S, kv_rows = (int64_t)pr.B * pr.Hkv * pr.S;
    if (!encode_rows_bf16(&mq, pr.q, q_rows, pr.D) ||
        !encode_rows_bf16(&mdo, pr.dout, q_rows, pr.D) ||
        !encode_rows_bf16(&mk, pr.k, kv_rows, pr.D) || !encode_rows_bf16(&mv, pr.v, kv_rows, pr.D))
        return RA_ERR_CUDA;
    Params P;
    const int Sb = (int)(pr.S / pr.N);
    const int nt = (Sb + kT - 1) / kT;
    P.G = make_tile_geom(pr.B, pr.Hq, pr.Hkv, pr.N, nt, pr.causal, pr.striped, which == 1);
    P.S = pr.S;
    P.Sb = Sb;
    P.rem = Sb - (nt - 1) * kT;
    P.sl2 = (float)((double)pr.scale * 1.4426950408889634);
    P.scale = pr.scale;
    P.lse = pr.lse;
    P.delta = pr.delta;
    P.dq = static_cast<__nv_bfloat16*>(pr.dq);
    P.dk = static_cast<__nv_bfloat16*>(pr.dk);
    P.dv = static_cast<__nv_bfloat16*>(pr.dv);
    P.status = status;
    P.work = work;
    P.timeout_cycles = timeout_cycles > 0 ? timeout_cycles : kTimeoutCycles;
    if (P.G.n_items <= 0) return RA_OK;
    if (cudaMemsetAsync(work, 0, sizeof(unsigned int), stream) != cudaSuccess) return RA_ERR_CUDA;
    const bool st = timeout_cycles > 0;
    auto kern = pr.D == 64
                    ? (which ? (st ? dkv_kernel<64, true> : dkv_kernel<64, false>)
                             : (st ? dq_kernel<64, true> : dq_kernel<64, false>))
                    : (which ? (st ? dkv_kernel<128, true> : dkv_kernel<128, false>)
                             : (st ? dq_kernel<128, true> : dq_kernel<128, false>));
    const int smem = which ? dkv::kSmemBytes : dqk::kSmemBytes;
    const long long grid = P.G.n_items < sm_count ? P.G.n_items : sm_count;
    if (which == 0 && !st && dq_from_last(P.G, grid, Sb, pr.D, l2_bytes_of_device()))
        kern = pr.D == 64 ? dq_kernel<64, false, false, true> : dq_kernel<128, false, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return RA_ERR_CUDA;
    kern<<<(unsigned)grid, kThreads, smem, stream>>>(mq, mdo, mk, mv, P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

// One ring step (see Params): the dq kernel over the shard's query tiles,
// then the dk/dv kernel over the block's key tiles, both STEP variants.
static int launch_step(const BwdStepProblem& pr, int which, unsigned int* status,
                       unsigned int* work, int sm_count, cudaStream_t stream) {
    CUtensorMap mq, mdo, mk, mv;
    const int64_t q_rows = (int64_t)pr.B * pr.Hq * pr.Sb, kv_rows = (int64_t)pr.B * pr.Hkv * pr.Sb;
    if (!encode_rows_bf16(&mq, pr.q, q_rows, pr.D) ||
        !encode_rows_bf16(&mdo, pr.dout, q_rows, pr.D) ||
        !encode_rows_bf16(&mk, pr.k, kv_rows, pr.D) || !encode_rows_bf16(&mv, pr.v, kv_rows, pr.D))
        return RA_ERR_CUDA;
    Params P = {};
    const int Sb = (int)pr.Sb;
    const int nt = (Sb + kT - 1) / kT;
    // items: the buffers' one shard (query tiles, resp. key tiles of the block)
    P.G = make_tile_geom(pr.B, pr.Hq, pr.Hkv, 1, nt, pr.causal, pr.layout, which == 1);
    P.S = Sb;
    P.Sb = Sb;
    P.rem = Sb - (nt - 1) * kT;
    P.sl2 = (float)((double)pr.scale * 1.4426950408889634);
    P.scale = pr.scale;
    P.lse = pr.lse;
    P.delta = pr.delta;
    P.dq = static_cast<__nv_bfloat16*>(pr.dq);
    P.dk = static_cast<__nv_bfloat16*>(pr.dk);
    P.dv = static_cast<__nv_bfloat16*>(pr.dv);
    P.status = status;
    P.work = work;
    P.timeout_cycles = kTimeoutCycles;
    P.ring.N = pr.N;
    P.ring.nt = nt;
    P.ring.causal = pr.causal;
    P.ring.striped = pr.layout;
    P.step_i = pr.i;
    P.step_j = pr.j;
    P.step_first = pr.first;
    P.step_last = pr.last;
    P.dq_state = pr.dq_state;
    P.dk_state = pr.dk_state;
    P.dv_state = pr.dv_state;
    if (P.G.n_items <= 0) return RA_OK;
    if (cudaMemsetAsync(work, 0, sizeof(unsigned int), stream) != cudaSuccess) return RA_ERR_CUDA;
    auto kern = pr.D == 64 ? (which ? dkv_kernel<64, false, true> : dq_kernel<64, false, true>)
                           : (which ? dkv_kernel<128, false, true> : dq_kernel<128, false, true>);
    const int smem = which ? dkv::kSmemBytes : dqk::kSmemBytes;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return RA_ERR_CUDA;
    const long long grid = P.G.n_items < sm_count ? P.G.n_items : sm_count;
    kern<<<(unsigned)grid, kThreads, smem, stream>>>(mq, mdo, mk, mv, P);
    return cudaGetLastError() == cudaSuccess ? RA_OK : RA_ERR_CUDA;
}

}  // namespace tcb

bool tc_bwd_step_supported(const BwdStepProblem& p) {
    if (p.D != 64 && p.D != 128) return false;
    if (p.Sb <= 0 || p.Sb > (1ll << 30)) return false;
    if (p.layout == kZigzag && p.Sb % (2 * tcb::kT)) return false;
    if ((int64_t)p.B * p.Hq * p.Sb >= (1ll << 31) || (int64_t)p.B * p.Hkv * p.Sb >= (1ll << 31))
        return false;
    return true;
}

int launch_bwd_tc_step(const BwdStepProblem& p, unsigned int* status, unsigned int* work,
                       int sm_count, cudaStream_t stream) {
    if (!tc_bwd_step_supported(p)) return RA_ERR_UNSUPPORTED;
    if (!work) return RA_ERR_INVALID_ARG;
    if (p.first) {
        // delta = rowsum(dout * out) of the shard, kept by the caller for the
        // later steps
        BwdProblem d = {};
        d.out = p.out;
        d.dout = p.dout;
        d.delta = p.delta;
        d.B = p.B;
        d.Hq = p.Hq;
        d.Hkv = p.Hkv;
        d.S = p.Sb;
        d.D = p.D;
        d.N = 1;
        d.dtype = RA_BF16;
        int rc = launch_bwd_delta(d, stream);
        if (rc) return rc;
    }
    // both kernels take items from the same counter, zeroed before each launch
    int rc = tcb::launch_step(p, 0, status, work, sm_count, stream);
    if (rc) return rc;
    return tcb::launch_step(p, 1, status, work, sm_count, stream);
}

bool tc_bwd_supported(const BwdProblem& p) {
    if (p.dtype != RA_BF16 || (p.D != 64 && p.D != 128)) return false;
    if (p.S % p.N) return false;
    const int64_t Sb = p.S / p.N;
    if (p.striped == kZigzag && Sb % (2 * tcb::kT)) return false;
    if (Sb > (1ll << 30)) return false;
    if ((int64_t)p.B * p.Hq * p.S >= (1ll << 31) || (int64_t)p.B * p.Hkv * p.S >= (1ll << 31))
        return false;
    return true;
}

int launch_bwd_tc_selftest(const BwdProblem& p, unsigned int* status, unsigned int* work,
                           int sm_count, cudaStream_t stream, long long timeout_cycles, int which) {
    if (!tc_bwd_supported(p)) return RA_ERR_UNSUPPORTED;
    if (!work || timeout_cycles <= 0 || (which != 0 && which != 1)) return RA_ERR_INVALID_ARG;
    return tcb::launch_one(p, which, status, work, sm_count, stream, timeout_cycles);
}

int launch_bwd_tc(const BwdProblem& p, unsigned int* status, unsigned int* work, int sm_count,
                  cudaStream_t stream) {
    if (!tc_bwd_supported(p)) return RA_ERR_UNSUPPORTED;
    if (!work) return RA_ERR_INVALID_ARG;
    // both kernels take items from the same counter, zeroed before each launch
    int rc = tcb::launch_one(p, 0, status, work, sm_count, stream);
    if (rc) return rc;
    return tcb::launch_one(p, 1, status, work, sm_count, stream);
}

}  // namespace ra
