"""Host-side shared-memory plans of the streaming GEMV (csrc/ggq_plan.h), on CPU.

The plan decides, per (format, tokens, K), between whole-row stages, row
chunks and running the tokens in groups.  A small host program compiled with
nvcc against the library's own header walks every format, every token count
1-8 and every K (multiples of 256 up to past the largest plan) the way the
pooled entry point recurses, and checks the invariants the kernel relies on:
the plan fits in the opt-in shared memory, a chunk is a whole number of its
format's granules and its byte count matches its units, row slots keep the
16-byte offset of an unaligned row, a stage holds 16 row slots, chunks give
every lane a unit when more than one token shares them, and splitting the
tokens never changes whether a shape can run (every token count runs exactly
the K that one token runs, up to the same bound).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gguf_block_quant_ggq_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "ggq_plan.h"
using namespace ggq;

static long violations = 0;
#define CHECK(c, ...) do { if (!(c)) { if (violations++ < 20) { std::printf(__VA_ARGS__); std::printf("\n"); } } } while (0)

static int64_t row_bytes(int f, int K) { return static_cast<int64_t>(K) / fmt_qk(f) * fmt_bytes(f); }

// bytes of u 64-weight units of format f (u a multiple of 4 for the 256-blocks)
static int64_t units_bytes(int f, int u) {
    if (fmt_qk(f) == 256) return static_cast<int64_t>(u / 4) * fmt_bytes(f);
    return static_cast<int64_t>(u) * 2 * fmt_bytes(f);
}

struct Counts { long runs = 0, chunked = 0, splits = 0; };

// The pooled entry point's recursion over token groups; false if a group has no plan.
static bool walk(int f, int T, int K, Counts& c) {
    const bool q81 = f == F_Q4_0;
    const int64_t rb = row_bytes(f, K);
    StreamShape sh;
    int cu = -1, cb = -1, rs = -1;
    const StreamPlan p = plan_gemv_stream(f, rb, T, K, q81, &sh, &cu, &cb, &rs);
    if (p == StreamPlan::kNone) return false;
    if (p == StreamPlan::kSplit) {
        ++c.splits;
        CHECK(T > 1, "split of one token f=%d K=%d", f, K);
        return walk(f, T / 2, K, c) && walk(f, T - T / 2, K, c);
    }
    ++c.runs;
    CHECK(sh.smem <= kSmemLimit, "smem %d > limit f=%d T=%d K=%d", sh.smem, f, T, K);
    CHECK(sh.stages >= 1 && sh.stages <= kMaxStages, "stages %d f=%d T=%d K=%d", sh.stages, f, T, K);
    CHECK(sh.x_bytes == x_region_bytes(T, K, q81), "x region f=%d T=%d K=%d", f, T, K);
    CHECK(sh.stride % 128 == 0, "stride %d not a multiple of 128", sh.stride);
    CHECK(sh.smem >= sh.stages * sh.stride + sh.x_bytes + 2 * kMaxStages * 8, "layout does not fit its plan");
    if (cu == 0) {  // whole rows: one stage holds a 16-row tile
        CHECK(cb == 0 && rs == 0, "whole-row plan with chunk fields");
        CHECK(sh.stride >= kTileRows * rb + 16, "whole-row stage too small f=%d K=%d", f, K);
        CHECK(sh.stages >= 2 || T == 1, "single whole-row stage for %d tokens f=%d K=%d", T, f, K);
        return true;
    }
    ++c.chunked;
    const int nu = units_per_row(K);
    int gu = 0, gb = 0;
    chunk_granule(f, rb, &gu, &gb);
    const bool small = f == F_Q6_K && cu % 32 != 0;  // the one-superblock granule of Q6_K
    if (small) gu = 4, gb = 210;
    CHECK(cu > 0 && cu % gu == 0 && cb == cu / gu * gb, "chunk %d units / %d bytes vs granule %d/%d f=%d K=%d",
          cu, cb, gu, gb, f, K);
    CHECK(cb == units_bytes(f, cu), "chunk bytes %d for %d units f=%d", cb, cu, f);
    CHECK(T == 1 || cu >= 32, "chunk of %d units shared by %d tokens f=%d K=%d", cu, T, f, K);
    CHECK(sh.stages >= 2, "chunked plan with %d stages", sh.stages);
    CHECK(rs % 16 == 0, "row slot %d not a multiple of 16", rs);
    const bool aligned = rb % 16 == 0 && cb % 16 == 0;
    CHECK(aligned ? rs >= cb : rs >= cb + 15, "row slot %d for chunk %d (aligned %d) f=%d K=%d", rs, cb, aligned, f, K);
    CHECK(sh.stride >= kTileRows * rs + 16, "stage %d < 16 row slots of %d", sh.stride, rs);
    const int nkc = (nu + cu - 1) / cu;
    const int64_t last = rb - static_cast<int64_t>(nkc - 1) * cb;
    CHECK(last > 0 && last <= cb, "last chunk %lld bytes (chunk %d, row %lld)", (long long)last, cb, (long long)rb);
    return true;
}

int main() {
    const int fmts[] = {F_Q4_0, F_Q8_0, F_MXFP4, F_Q4_K, F_Q5_K, F_Q6_K};
    for (int f : fmts) {
        Counts c;
        int max_one = 0;
        bool ended = false;
        for (int K = 256; K <= 160000; K += 256) {
            const bool one = walk(f, 1, K, c);
            if (one) {
                CHECK(!ended, "f=%d: K=%d runs after a smaller K did not", f, K);
                max_one = K;
            } else {
                ended = true;
            }
            for (int T = 2; T <= 8; ++T) CHECK(walk(f, T, K, c) == one, "f=%d T=%d K=%d differs from one token", f, T, K);
        }
        std::printf("fmt %d max_k %d runs %ld chunked %ld splits %ld\n", f, max_one, c.runs, c.chunked, c.splits);
    }
    std::printf("violations %ld\n", violations);
    return violations == 0 ? 0 : 1;
}
"""


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_streaming_plans_keep_their_invariants(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    src = tmp_path / "plan_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "plan_check"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    lines = dict((ln.split()[1], ln) for ln in r.stdout.splitlines() if ln.startswith("fmt "))
    # every format runs K up to 146432 (the bound stated for ggq_mul_mat_vec)
    for ln in lines.values():
        assert int(ln.split()[3]) >= 146432, ln
    assert "violations 0" in r.stdout
