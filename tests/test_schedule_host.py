"""Host checks of the forward kernel's fold walk (no GPU): the schedule header
compiled as plain C++ with g++.  Entered at a common block (TileWalkFromLast),
a query tile's walk must fold exactly the tiles of its ring-order walk, as
the same cyclic order rotated; the host rule that turns the common entry on
keeps the ring order whenever the concurrently read key/value shards fit in
L2."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_long_context_order_b300", "csrc")

HARNESS = r"""
#define RA_HD inline
#include "schedule.cuh"
#include <cstdio>
#include <cstdlib>
#include <vector>
using namespace ra;

struct F { int s, j, kt; };

template <class W>
static std::vector<F> walk(const ItemGeom& G, const Item& it) {
    std::vector<F> v;
    W w;
    for (w.start(G.rg, it); !w.done(G.rg); w.next(G.rg, it)) v.push_back({w.s, w.j, w.kt});
    return v;
}

// For every item: the walk entered at block N-1 visits key shards N-1, N-2,
// ..., 0 and equals the ring-order walk's steps rotated to start at step
// (i + 1) mod N, each step with the same key tiles in the same order, and
// s = (i - j) mod N throughout.
static int check(int B, int Hq, int Hkv, int N, int nt, int causal, int layout) {
    const ItemGeom G = make_item_geom(B, Hq, Hkv, N, nt, causal, layout);
    for (long long item = 0; item < G.n_items; ++item) {
        const Item it = decode_item(G, item);
        const std::vector<F> a = walk<TileWalk>(G, it);
        const int s0 = (it.i + 1) % N;
        const std::vector<F> b = walk<TileWalkFromLast>(G, it);
        if (a.size() != b.size()) return 1;
        // a's entries from step s0 on, then those before it
        std::vector<F> r;
        for (const F& f : a) if (f.s >= s0) r.push_back(f);
        for (const F& f : a) if (f.s < s0) r.push_back(f);
        int prev_j = N;
        for (size_t k = 0; k < b.size(); ++k) {
            if (b[k].s != r[k].s || b[k].j != r[k].j || b[k].kt != r[k].kt) return 2;
            if (((it.i - b[k].j) % N + N) % N != b[k].s) return 3;
            if (b[k].j > prev_j) return 4;
            prev_j = b[k].j;
        }
    }
    return 0;
}

int main(int argc, char** argv) {
    if (argc == 8) {
        printf("%d\n", check(atoi(argv[1]), atoi(argv[2]), atoi(argv[3]), atoi(argv[4]),
                             atoi(argv[5]), atoi(argv[6]), atoi(argv[7])));
        return 0;
    }
    // ring_entry: B Hq Hkv N nt causal layout grid Sb D l2
    if (argc == 12) {
        ItemGeom G = make_item_geom(atoi(argv[1]), atoi(argv[2]), atoi(argv[3]), atoi(argv[4]),
                                    atoi(argv[5]), atoi(argv[6]), atoi(argv[7]));
        printf("%d\n", ring_entry(G, atoll(argv[8]), atoi(argv[9]), atoi(argv[10]),
                                  atoll(argv[11])));
        return 0;
    }
    return 1;
}
"""


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("sched")
    src, exe = d / "h.cpp", d / "h"
    src.write_text(HARNESS)
    subprocess.run([cxx, "-std=c++17", "-O2", "-x", "c++", f"-I{CSRC}", str(src), "-o", str(exe)],
                   check=True)

    def run(*args):
        r = subprocess.run([str(exe)] + [str(a) for a in args], capture_output=True, text=True,
                           check=True)
        return int(r.stdout.strip())
    return run


# (B, Hq, Hkv, N, nt, causal, layout): paired heads (even group), odd groups
# (paired query tiles, odd nt), striped, zigzag and non-causal
GEOMS = [
    (1, 8, 1, 8, 6, 1, 1),
    (1, 8, 1, 6, 10, 1, 2),
    (2, 4, 2, 4, 7, 1, 1),
    (1, 3, 1, 5, 9, 1, 1),
    (1, 3, 3, 4, 6, 1, 2),
    (2, 2, 1, 3, 5, 0, 0),
    (1, 2, 1, 7, 4, 0, 1),
]


@pytest.mark.parametrize("geom", GEOMS)
def test_common_entry_is_the_ring_walk_rotated(harness, geom):
    assert harness(*geom) == 0, geom


L2 = 126 * 1000 * 1000


@pytest.mark.parametrize("name,args,want", [
    # 128K tokens, 32 query heads on 8 KV heads, 16 shards of 8192: the 16
    # shards' keys and values (64 MiB per KV head) fit, ring order
    ("gqa_128k", (1, 32, 8, 16, 64, 1, 1, 148, 8192, 128), 0),
    ("gqa_128k_ragged", (1, 32, 8, 16, 63, 1, 1, 148, 8000, 128), 0),
    ("causal_32k_striped", (2, 32, 32, 8, 32, 1, 1, 148, 4096, 128), 0),
    ("causal_32k_zigzag", (2, 32, 32, 8, 32, 1, 2, 148, 4096, 128), 0),
    ("noncausal_8k", (1, 8, 8, 8, 8, 0, 0, 148, 1024, 128), 0),
    # 1M tokens, 8 query heads on one KV head, 64 shards of 16384: the grid
    # holds 37 query shards reading 37 blocks of 8 MiB at once
    ("long_1m", (1, 8, 1, 64, 128, 1, 1, 148, 16384, 128), 1),
    # 2 query heads on one KV head, 16 shards of 24576: 16 blocks of 24 MiB
    ("long_shards_384k", (1, 2, 1, 16, 192, 1, 1, 148, 24576, 128), 1),
    # contiguous causal keeps its own order (global query tiles)
    ("long_1m_contiguous", (1, 8, 1, 64, 128, 1, 0, 148, 16384, 128), 0),
])
def test_ring_entry_rule(harness, name, args, want):
    assert harness(*args, L2) == want, name


def test_bench_names_the_kernel_the_rule_picks(harness):
    """bench.py reports the forward instantiation by restating the host rule
    in Python; for every named workload it must agree with ring_entry."""
    import bench
    import ragen
    sms = 148
    for name, wl in ragen.WORKLOADS.items():
        if wl.dtype != "bf16":
            continue
        Sb = wl.S // wl.N
        nt = (Sb + 127) // 128
        g = wl.Hq // wl.Hkv
        items = wl.B * wl.Hkv * wl.N * ((g // 2) * nt if g % 2 == 0 else g * ((nt + 1) // 2))
        kname = bench.kernel_name(wl, sms, L2)
        if "kModeStreamK" in kname:
            continue
        want = harness(wl.B, wl.Hq, wl.Hkv, wl.N, nt, int(wl.causal), int(wl.striped),
                       min(items, sms), Sb, wl.D, L2)
        assert ("kModeRingFromLast" in kname) == bool(want), name
