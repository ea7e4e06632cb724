"""The work split of the kernels (body + shared tail, `lin_attn_internal.cuh`), checked on
the host: a small program built from the same header walks every split the library can
make for a range of shapes and checks that

  * the chunks' virtual ranges partition the layer's (head, tile) pairs exactly once;
  * every run of a chunk stays in one head and covers consecutive tiles;
  * the KV plan's partial slots of a head are distinct, dense and within its budget, and
    the bound used to size scratch is never exceeded;
  * a launch over a subset of heads (the host-buffer path's pipeline) does the same
    segments, tile for tile, as the whole-layer launch (so its sums are bitwise the same);
  * a tail is only used where it shortens the costliest chunk (tiles plus a switch cost per
    extra head) below the longest chunk of the split without one.

No GPU is involved: the program only calls the header's host/device inline functions."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

CSRC = os.path.join(ROOT, "video_diffusion_dit_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "lin_attn_internal.cuh"
using namespace la;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { if (fails++ < 20) { std::printf(__VA_ARGS__); std::printf("\n"); } } } while (0)

// Partition, runs, 32-bit map and balance of one split.
static void check_split(const TileSplit& s, int ctas, const char* what, int64_t switch_cost) {
    const int64_t H = s.heads, T = s.tiles_per_head, total = H * T;
    CHECK(s.chunks == s.per_head * s.heads + s.tail_chunks, "%s: chunk count", what);
    CHECK(s.per_head >= 1 && s.body >= s.per_head && s.body <= T, "%s: k=%d B=%lld T=%lld", what, s.per_head,
          (long long)s.body, (long long)T);
    if (s.heads * s.per_head <= ctas) CHECK(s.chunks <= ctas, "%s: %d chunks > %d CTAs", what, s.chunks, ctas);
    CHECK(split_begin(s, 0) == 0 && split_begin(s, s.chunks) == total, "%s: ends", what);
    std::vector<int> seen(total, 0);
    int64_t worst = 0;  // tiles + switch_cost per head beyond the first, of the costliest chunk
    for (int c = 0; c < s.chunks; ++c) {
        const int64_t b = split_begin(s, c), e = split_begin(s, c + 1);
        CHECK(e > b, "%s: empty chunk %d", what, c);
        int64_t cost = (e - b) - switch_cost;
        for (int64_t v = b; v < e;) {
            cost += switch_cost;
            const int64_t r = split_run_end(s, v) < e ? split_run_end(s, v) : e;
            CHECK(r > v, "%s: run", what);
            const HeadTile first = split_tile(s, v);
            for (int64_t w = v; w < r; ++w) {
                const HeadTile x = split_tile(s, w);
                CHECK(x.h == first.h && x.tile == first.tile + (w - v), "%s: run of chunk %d not one head", what, c);
                CHECK(x.h >= 0 && x.h < H && x.tile >= 0 && x.tile < T, "%s: out of range", what);
                if (x.h >= 0 && x.h < H && x.tile >= 0 && x.tile < T) ++seen[x.h * T + x.tile];
                if (total < (int64_t(1) << 31)) {
                    int h32, t32;
                    split_tile32(s, static_cast<int>(w), h32, t32);
                    CHECK(h32 == x.h && t32 == x.tile, "%s: 32-bit map", what);
                }
            }
            v = r;
        }
        worst = cost > worst ? cost : worst;
    }
    for (int64_t i = 0; i < total; ++i) CHECK(seen[i] == 1, "%s: tile %lld covered %d times", what, (long long)i, seen[i]);
    // A tail is only taken where it makes the costliest chunk cheaper than the longest part
    // of the split without one.
    if (s.tail_chunks > 0)
        CHECK(worst < (T + s.per_head - 1) / s.per_head, "%s: costliest chunk %lld, without a tail %lld", what,
              (long long)worst, (long long)((T + s.per_head - 1) / s.per_head));
}

// Segments (chunk, head, first tile, end tile) a launch over heads [h0, h0 + hc) performs.
struct Seg { int64_t c; int h, slot; int64_t t0, t1; };
static std::vector<Seg> launch_segments(const KvPlan& p, int h0, int hc) {
    const KvLaunch w = kv_launch(p, h0, hc);
    std::vector<Seg> out;
    for (int b = 0; b < w.n_chunks; ++b) {
        int64_t c, ts, te;
        if (b < w.n_body) {
            c = w.c_body + b;
            ts = split_begin(p, c);
            te = split_begin(p, c + 1);
        } else {
            c = w.c_tail + (b - w.n_body);
            ts = split_begin(p, c) > w.tail_lo ? split_begin(p, c) : w.tail_lo;
            te = split_begin(p, c + 1) < w.tail_hi ? split_begin(p, c + 1) : w.tail_hi;
        }
        CHECK(te > ts, "launch h0=%d hc=%d: empty CTA %d", h0, hc, b);
        for (int64_t v = ts; v < te;) {
            const int64_t r = split_run_end(p, v) < te ? split_run_end(p, v) : te;
            const HeadTile x = split_tile(p, v);
            CHECK(x.h >= h0 && x.h < h0 + hc, "launch h0=%d hc=%d: head %d outside", h0, hc, x.h);
            out.push_back(Seg{c, x.h, segment_of(p, x.h, c), x.tile, x.tile + (r - v)});
            v = r;
        }
    }
    return out;
}

static void check_plan(int H, int64_t N) {
    char what[96];
    std::snprintf(what, sizeof what, "kv H=%d N=%lld", H, (long long)N);
    const KvPlan p = kv_plan(H, N);
    check_split(p, kChunks, what, kKvSwitchCost);
    CHECK(p.per_head <= kChunksPerHeadCap, "%s: k", what);
    CHECK(p.seg_stride <= kv_seg_stride_bound(H) && kv_seg_stride_bound(H) <= kMaxSegments, "%s: stride %d bound %d",
          what, p.seg_stride, kv_seg_stride_bound(H));
    const std::vector<Seg> all = launch_segments(p, 0, H);
    std::vector<std::vector<int>> slots(H);
    int most = 0;
    for (const Seg& s : all) {
        CHECK(s.slot >= 0 && s.slot < segments_of_head(p, s.h), "%s: slot %d of head %d", what, s.slot, s.h);
        slots[s.h].push_back(s.slot);
    }
    for (int h = 0; h < H; ++h) {
        const int n = segments_of_head(p, h);
        most = n > most ? n : most;
        CHECK(static_cast<int>(slots[h].size()) == n, "%s: head %d has %zu segments, expects %d", what, h,
              slots[h].size(), n);
        std::vector<int> hit(n, 0);
        for (int x : slots[h]) if (x >= 0 && x < n) ++hit[x];
        for (int i = 0; i < n; ++i) CHECK(hit[i] == 1, "%s: head %d slot %d used %d times", what, h, i, hit[i]);
    }
    CHECK(most == p.seg_stride, "%s: seg_stride %d, most %d", what, p.seg_stride, most);
    const int widths[] = {1, 2, (H + 19) / 20, 3};
    for (int hc : widths) {
        if (hc < 1 || hc > H) continue;
        std::vector<Seg> parts;
        for (int h0 = 0; h0 < H; h0 += hc) {
            const std::vector<Seg> q = launch_segments(p, h0, h0 + hc <= H ? hc : H - h0);
            parts.insert(parts.end(), q.begin(), q.end());
        }
        CHECK(parts.size() == all.size(), "%s: %zu segments by %d-head launches, %zu whole", what, parts.size(), hc,
              all.size());
        for (const Seg& a : all) {
            bool found = false;
            for (const Seg& b : parts)
                if (b.c == a.c && b.h == a.h && b.slot == a.slot && b.t0 == a.t0 && b.t1 == a.t1) found = true;
            CHECK(found, "%s: segment (chunk %lld, head %d) differs in %d-head launches", what, (long long)a.c, a.h, hc);
        }
    }
    CHECK(kv_launch(p, 0, H).n_chunks == p.chunks, "%s: whole launch CTAs", what);
}

int main() {
    const int heads[] = {1, 2, 3, 7, 10, 11, 12, 16, 19, 20, 24, 32, 40, 64, 76, 100, 151, 152, 153, 300};
    const int64_t tokens[] = {1, 63, 64, 65, 200, 640, 1000, 4096, 9728, 32760, 180320, 262144, 1000003};
    for (int H : heads)
        for (int64_t N : tokens) {
            if (H * N > 300000000) continue;
            check_plan(H, N);
            char what[96];
            const int64_t T = (N + kApplyTile - 1) / kApplyTile;
            for (int ctas : {152, 148, 132, 1}) {
                std::snprintf(what, sizeof what, "apply H=%d T=%lld G=%d", H, (long long)T, ctas);
                check_split(tile_split(H, T, ctas, kNoPerHeadCap, kApplyMinPart, kApplySwitchCost), ctas, what,
                            kApplySwitchCost);
                check_split(tile_split(H, T, ctas, kNoPerHeadCap, 0, 0), ctas, what, 0);
            }
            std::snprintf(what, sizeof what, "whole H=%d T=%lld", H, (long long)T);
            const TileSplit w = tile_split(H, T, H, 1, 0, 0);
            CHECK(w.tail_chunks == 0 && w.body == T, "%s: not whole heads", what);
        }
    // The shapes the kernels are measured on.
    const KvPlan p720 = kv_plan(20, 180320);
    CHECK(p720.chunks == 152 && p720.per_head == 7 && p720.tail_chunks == 12, "720p plan %d %d %d", p720.chunks,
          p720.per_head, p720.tail_chunks);
    const KvPlan pd64 = kv_plan(32, 180320);
    CHECK(pd64.chunks == 152 && pd64.per_head == 4 && pd64.tail_chunks == 24, "D=64 plan %d %d %d", pd64.chunks,
          pd64.per_head, pd64.tail_chunks);
    std::printf(fails ? "FAILED %d\n" : "OK\n", fails);
    return fails ? 1 : 0;
}
"""


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="needs nvcc to build the host program")
def test_work_split_partitions_and_plans(tmp_path):
    src = tmp_path / "split_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "split_check"
    r = subprocess.run(["nvcc", "-std=c++17", "-O2", "-I", CSRC, str(src), "-o", str(exe)], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
