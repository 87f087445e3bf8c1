// Ring fold schedule and persistent work decomposition, shared by the host
// planners (ra_plan, ra_plan_backward) and the kernels.
//
// Ring schedule ("Ring Attention" glossary page, "Como funciona a atencao em
// anel"): query shard i folds key/value shard j = (i - s) mod N at step s.
// Within a shard pair the key tiles are folded in ascending order.  With
// 128-token tiles and equal query/key tile sizes the causal mask reduces to a
// closed form per (i, j, qt, kt):
//   non-causal            every key tile of every shard, FULL
//   causal, contiguous    j < i: every key tile FULL; j == i: kt < qt FULL,
//                         kt == qt INCL (local key row <= local query row);
//                         j > i: nothing
//   causal, striped       (token t on shard t mod N, local row t div N): for
//                         every j, kt < qt FULL and kt == qt INCL if j <= i,
//                         STRICT (local key row < local query row) if j > i
// since token r*N + i sees token c*N + j iff c < r, or c == r and j <= i.
//   causal, zigzag        (2N chunks of Sb/2 tokens; shard i holds chunk i,
//                         then chunk 2N-1-i; h = nt/2 tiles per chunk): a
//                         query tile in the first half sees the first half of
//                         shards j < i and its own chunk up to the diagonal;
//                         one in the second half sees all of shards j > i,
//                         the first half of shards j < i, and its own shard up
//                         to the diagonal (INCL).  Live tiles are always a
//                         prefix [0, nk) of shard j.
#pragma once
#include <cstdint>

#ifndef RA_HD
#define RA_HD __host__ __device__ __forceinline__
#endif

namespace ra {

enum FoldKind : int { kFull = 0, kIncl = 1, kStrict = 2, kNone = 3 };
enum Layout : int { kContiguous = 0, kStriped = 1, kZigzag = 2 };

struct RingGeom {
    int N;        // virtual devices (shards)
    int nt;       // tiles per shard (Sb / tile)
    int causal;
    int striped;  // layout: kContiguous, kStriped or kZigzag
};

// Live key tiles of shard j for query tile qt of shard i: kt in [0, *nk); the
// tile kt == qt (when *diag_kind != kNone) is the masked diagonal tile.
RA_HD void shard_span(const RingGeom& g, int i, int j, int qt, int* nk, int* diag_kind) {
    if (!g.causal) {
        *nk = g.nt;
        *diag_kind = kNone;
    } else if (g.striped == kContiguous) {
        if (j < i) { *nk = g.nt; *diag_kind = kNone; }
        else if (j == i) { *nk = qt + 1; *diag_kind = kIncl; }
        else { *nk = 0; *diag_kind = kNone; }
    } else if (g.striped == kStriped) {
        *nk = qt + 1;
        *diag_kind = (j <= i) ? kIncl : kStrict;
    } else {  // zigzag
        const int h = g.nt / 2;
        *diag_kind = kNone;
        if (j == i) { *nk = qt + 1; *diag_kind = kIncl; }
        else if (qt < h) *nk = (j < i) ? h : 0;
        else *nk = (j > i) ? g.nt : h;
    }
}

RA_HD int fold_kind(const RingGeom& g, int i, int j, int qt, int kt) {
    int nk, dk;
    shard_span(g, i, j, qt, &nk, &dk);
    if (kt >= nk) return kNone;
    return (kt == qt && dk != kNone) ? dk : kFull;
}

// Query tiles of shard i that see key tile kt of shard j: qt in [*q_lo, *q_hi).
// The transpose of shard_span: for every (i, j, qt, kt), qt lies in the range
// exactly when fold_kind(g, i, j, qt, kt) != kNone.
RA_HD void key_span(const RingGeom& g, int i, int j, int kt, int* q_lo, int* q_hi) {
    *q_lo = 0;
    *q_hi = g.nt;
    if (!g.causal) return;
    if (g.striped == kContiguous) {
        if (j == i) *q_lo = kt;
        else if (j > i) *q_hi = 0;
        return;
    }
    if (g.striped == kStriped) {
        *q_lo = kt;
        return;
    }
    const int h = g.nt / 2;  // zigzag
    if (j == i) *q_lo = kt;
    else if (j < i) { if (kt >= h) *q_hi = 0; }
    else *q_lo = h;
}

// Work items of the backward kernels, one 128-row tile each, numbered group
// major ((b, kv head) outer) and, inside a group, longest work first.
//  * query tiles (dq kernel): the fold list of (i, qt); within a group,
//    index lam * W + w with lam the cost level (as for the forward) and w the
//    query head and shard;
//  * key tiles (dk/dv kernel): the transposed list of (j, kt), visited by
//    every query head of the group.  Cost of (j, kt) in live query tiles:
//    non-causal and striped N*nt resp. N*(nt - kt) (order kt, then j);
//    contiguous (N-1-j)*nt + nt - kt (order j, then kt); zigzag (h = nt/2)
//    N*nt - (j*h + kt) for kt < h, then j*h + nt - kt for kt >= h.
struct TileGeom {
    RingGeom rg;
    int B, Hq, Hkv, g;
    long long per_group;  // items per (b, kv head)
    long long n_items;
};

RA_HD TileGeom make_tile_geom(int B, int Hq, int Hkv, int N, int nt, int causal, int striped,
                              bool key_tiles) {
    TileGeom G;
    G.rg.N = N; G.rg.nt = nt; G.rg.causal = causal; G.rg.striped = striped;
    G.B = B; G.Hq = Hq; G.Hkv = Hkv; G.g = Hq / Hkv;
    G.per_group = (long long)N * nt * (key_tiles ? 1 : G.g);
    G.n_items = (long long)B * Hkv * G.per_group;
    return G;
}

struct QTile {
    int b, kvh, h, i, qt;
};

RA_HD QTile decode_qtile(const TileGeom& G, long long item) {
    QTile t;
    const long long grp = item / G.per_group, rem = item % G.per_group;
    t.b = (int)(grp / G.Hkv);
    t.kvh = (int)(grp % G.Hkv);
    const int N = G.rg.N, nt = G.rg.nt;
    if (G.rg.causal && G.rg.striped == kContiguous) {
        const int lam = (int)(rem / G.g), w = (int)(rem % G.g);
        const int gt = N * nt - 1 - lam;
        t.i = gt / nt;
        t.qt = gt % nt;
        t.h = t.kvh * G.g + w;
    } else {
        const int W = N * G.g;
        const int lam = (int)(rem / W), w = (int)(rem % W);
        t.qt = nt - 1 - lam;
        t.i = w / G.g;
        t.h = t.kvh * G.g + w % G.g;
    }
    return t;
}

struct KTile {
    int b, kvh, j, kt;
};

RA_HD KTile decode_ktile(const TileGeom& G, long long item) {
    KTile t;
    const long long grp = item / G.per_group;
    const int e = (int)(item % G.per_group);
    t.b = (int)(grp / G.Hkv);
    t.kvh = (int)(grp % G.Hkv);
    const int N = G.rg.N, nt = G.rg.nt;
    if (G.rg.causal && G.rg.striped == kContiguous) {
        t.j = e / nt;
        t.kt = e % nt;
    } else if (G.rg.causal && G.rg.striped == kZigzag) {
        const int h = nt / 2;
        if (e < N * h) {
            t.j = e / h;
            t.kt = e % h;
        } else {
            const int e2 = e - N * h;
            t.j = N - 1 - e2 / h;
            t.kt = h + e2 % h;
        }
    } else {
        t.kt = e / N;
        t.j = e % N;
    }
    return t;
}

// Visiting order of the dk/dv kernel for key tile kt of shard j.  The block
// and its gradient accumulators go round the ring in its cyclic order, but
// every block enters it at device 0 rather than at its own device j: query
// shards i = 0, 1, ..., N-1, where the block arrives at ring step
// s = (i - j) mod N.  Blocks running at the same time then read the same
// query shards while those are in L2.  Within a shard: the query heads of
// the GQA group (gi < heads), then the query tiles that see the key tile,
// ascending.  Shards with no such tile are skipped.
struct KeyWalk {
    int s, i, gi, qt, q_lo, q_hi;
    RA_HD void start(const RingGeom& g, int j, int kt, int heads) {
        i = -1;
        s = 0;
        advance_shard(g, j, kt);
        (void)heads;
    }
    RA_HD void advance_shard(const RingGeom& g, int j, int kt) {
        for (;;) {
            ++i;
            if (i >= g.N) return;
            s = i - j;
            if (s < 0) s += g.N;
            key_span(g, i, j, kt, &q_lo, &q_hi);
            if (q_lo < q_hi) {
                gi = 0;
                qt = q_lo;
                return;
            }
        }
    }
    RA_HD bool done(const RingGeom& g) const { return i >= g.N; }
    RA_HD void next(const RingGeom& g, int j, int kt, int heads) {
        if (++qt < q_hi) return;
        qt = q_lo;
        if (++gi < heads) return;
        advance_shard(g, j, kt);
    }
};

// Persistent work items of the tensor-core kernel.  An item is two 128-row
// query tiles ("slots") that share every key/value tile they stream:
//  * pair_heads = 1 (Hq/Hkv even): query heads 2m and 2m+1 of one GQA group at
//    the same query tile -- identical fold lists;
//  * pair_heads = 0: query tiles 2p and 2p+1 of one head -- slot 0 treats the
//    extra diagonal tile of slot 1 as fully masked (kNone).
// Items are numbered group-major ((b, kv head) outer), then by "level" in
// decreasing cost (longest work first), then within a level.
struct ItemGeom {
    RingGeom rg;
    int B, Hq, Hkv, g;
    int pair_heads;
    int L, W;  // levels per group, items per level
    long long n_items;
};

RA_HD ItemGeom make_item_geom(int B, int Hq, int Hkv, int N, int nt, int causal, int striped) {
    ItemGeom G;
    G.rg.N = N; G.rg.nt = nt; G.rg.causal = causal; G.rg.striped = striped;
    G.B = B; G.Hq = Hq; G.Hkv = Hkv; G.g = Hq / Hkv;
    G.pair_heads = (G.g % 2 == 0) ? 1 : 0;
    const bool contig_causal = causal && striped == kContiguous;
    if (G.pair_heads) {
        int hp = G.g / 2;
        G.L = contig_causal ? N * nt : nt;
        G.W = contig_causal ? hp : N * hp;
    } else {
        int nt2 = (nt + 1) / 2;
        G.L = contig_causal ? N * nt2 : nt2;
        G.W = contig_causal ? G.g : N * G.g;
    }
    G.n_items = (long long)B * Hkv * G.L * G.W;
    return G;
}

// Whether the forward's query shards enter the ring at a common block
// (TileWalkFromLast; host side).  In ring order the `grid` CTAs running
// together hold items of about grid / per_shard query shards, and at a moment
// each of these folds a different key/value shard (shard i folds i - s at
// step s), so a block read by query shard i is wanted again by shard i + 1
// one step later.  When those blocks' keys and values (4 * Sb * D bytes per
// KV head) exceed the L2 they are evicted in between and every query shard
// reads them from DRAM again.  Entered at block N-1, all query shards of a
// level fold the same block at the same time (their steps have equal length
// whenever the fold kind does not depend on j: striped and non-causal).  On
// one GPU every block is resident from the start, so the entry point is free;
// the fold order stays a rotation of the ring's cyclic order.
inline int ring_entry(const ItemGeom& G, long long grid, int Sb, int D, long long l2_bytes) {
    const bool contig_causal = G.rg.causal && G.rg.striped == kContiguous;
    if (contig_causal || G.rg.N <= 1 || l2_bytes <= 0 || grid <= 0) return 0;
    const long long per_shard = G.W / G.rg.N;
    long long shards = (grid + per_shard - 1) / per_shard;
    if (shards > G.rg.N) shards = G.rg.N;
    return (double)shards * 4.0 * Sb * D > (double)l2_bytes ? 1 : 0;
}

struct Item {
    int b, kvh, i;
    int h[2], qt[2];
    int valid1;  // slot 1 holds a real query tile
};

RA_HD Item decode_item(const ItemGeom& G, long long item) {
    Item it;
    long long per_group = (long long)G.L * G.W;
    long long grp = item / per_group, rem = item % per_group;
    int lam = (int)(rem / G.W), w = (int)(rem % G.W);
    it.b = (int)(grp / G.Hkv);
    it.kvh = (int)(grp % G.Hkv);
    const int N = G.rg.N, nt = G.rg.nt;
    const bool contig_causal = G.rg.causal && G.rg.striped == kContiguous;
    if (G.pair_heads) {
        int hp_count = G.g / 2, hp, qt;
        if (contig_causal) {
            int gt = N * nt - 1 - lam;
            it.i = gt / nt; qt = gt % nt; hp = w;
        } else {
            qt = nt - 1 - lam; it.i = w / hp_count; hp = w % hp_count;
        }
        it.h[0] = it.kvh * G.g + 2 * hp;
        it.h[1] = it.h[0] + 1;
        it.qt[0] = it.qt[1] = qt;
        it.valid1 = 1;
    } else {
        int nt2 = (nt + 1) / 2, p, hh;
        if (contig_causal) {
            int gp = N * nt2 - 1 - lam;
            it.i = gp / nt2; p = gp % nt2; hh = w;
        } else {
            p = nt2 - 1 - lam; it.i = w / G.g; hh = w % G.g;
        }
        it.h[0] = it.h[1] = it.kvh * G.g + hh;
        it.qt[0] = 2 * p;
        it.qt[1] = 2 * p + 1;
        it.valid1 = (2 * p + 1 < nt) ? 1 : 0;
        if (!it.valid1) it.qt[1] = it.qt[0];  // slot 1 recomputes slot 0's tile, never stored
    }
    return it;
}

// Walks the union fold list of an item: ring steps s ascending, key tiles of
// shard j = (i - s) mod N ascending, over the key tiles either slot needs.
struct TileWalk {
    int s, j, kt, nk;
    RA_HD void start(const RingGeom& g, const Item& it) {
        s = -1; kt = 0; nk = 0; j = it.i;
        advance_shard(g, it);
    }
    RA_HD void advance_shard(const RingGeom& g, const Item& it) {
        // move to the next ring step with at least one live key tile
        for (;;) {
            ++s;
            if (s >= g.N) return;
            j = it.i - s;
            if (j < 0) j += g.N;
            int nk0, nk1, d;
            shard_span(g, it.i, j, it.qt[0], &nk0, &d);
            shard_span(g, it.i, j, it.qt[1], &nk1, &d);
            nk = nk0 > nk1 ? nk0 : nk1;
            kt = 0;
            if (nk > 0) return;
        }
    }
    RA_HD bool done(const RingGeom& g) const { return s >= g.N; }
    RA_HD void next(const RingGeom& g, const Item& it) {
        if (++kt >= nk) advance_shard(g, it);
    }
};

// The same fold list entered at a common block (ring_entry): key shards
// j = N-1, N-2, ..., 0, i.e. ring steps s = (i - j) mod N from (i + 1) mod N
// cyclically, each shard's live key tiles ascending.
struct TileWalkFromLast {
    int s, j, kt, nk;
    RA_HD void start(const RingGeom& g, const Item& it) {
        j = g.N; s = 0; kt = 0; nk = 0;
        advance_shard(g, it);
    }
    RA_HD void advance_shard(const RingGeom& g, const Item& it) {
        for (;;) {
            if (--j < 0) return;
            s = it.i - j;
            if (s < 0) s += g.N;
            int nk0, nk1, d;
            shard_span(g, it.i, j, it.qt[0], &nk0, &d);
            shard_span(g, it.i, j, it.qt[1], &nk1, &d);
            nk = nk0 > nk1 ? nk0 : nk1;
            kt = 0;
            if (nk > 0) return;
        }
    }
    RA_HD bool done(const RingGeom&) const { return j < 0; }
    RA_HD void next(const RingGeom& g, const Item& it) {
        if (++kt >= nk) advance_shard(g, it);
    }
};

}  // namespace ra
