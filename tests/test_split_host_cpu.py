"""Host-side arithmetic of the decode GEMMs' cluster split-K (CPU only): the
K split of a slab's k-blocks over the CTAs of a cluster, the output rows each
CTA owns and reduces, the push receive-buffer size, and the split-count
choice.  The helpers are the ones the kernels use (decode_common.cuh),
compiled here as host code by nvcc; nothing runs on a GPU."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

CSRC = os.path.join(ROOT, "fp8_w8a8_quantized_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "decode_common.cuh"
using namespace fp8k::decode;

static int fails = 0;
#define CHECK(c, ...) do { if (!(c)) { ++fails; std::printf(__VA_ARGS__); std::printf("\n"); } } while (0)

int main() {
    for (int S = 1; S <= kMaxSplits; ++S) {
        // owners: whole 4-row groups, contiguous, covering the 128-row slab,
        // none empty
        const int rp = owner_rows(S);
        CHECK(rp % 4 == 0, "S=%d owner_rows=%d not a multiple of 4", S, rp);
        int covered = 0;
        for (int rank = 0; rank < S; ++rank) {
            const int lo = rank * rp;
            const int hi = lo + rp < BNW ? lo + rp : BNW;
            const int width = hi > lo ? hi - lo : 0;
            CHECK(lo == covered, "S=%d rank %d starts at %d, expected %d", S, rank, lo, covered);
            CHECK(width > 0 && width % 4 == 0, "S=%d rank %d width %d", S, rank, width);
            covered += width;
        }
        CHECK(covered == BNW, "S=%d owners cover %d rows", S, covered);
        // push receive buffer: [S][rows_per][stride] fp32 fits for every M
        for (int M = 1; M <= 64; ++M) {
            const long need = static_cast<long>(S) * rp * push_stride(M) * 4;
            CHECK(push_recv_bytes(M, S) >= need && push_recv_bytes(M, S) % 128 == 0,
                  "S=%d M=%d recv %u < %ld", S, M, push_recv_bytes(M, S), need);
            CHECK(push_stride(M) >= M && push_stride(M) % 4 == 0, "stride M=%d", M);
        }
        // K split: contiguous slices covering every k-block, sizes differ by <= 1
        for (int nk = S; nk <= 300; ++nk) {
            int next = 0, mn = 1 << 30, mx = 0;
            for (int rank = 0; rank < S; ++rank) {
                int kb0, nkb;
                split_range(rank, nk, S, &kb0, &nkb);
                CHECK(kb0 == next, "nk=%d S=%d rank %d kb0 %d", nk, S, rank, kb0);
                next = kb0 + nkb;
                mn = nkb < mn ? nkb : mn;
                mx = nkb > mx ? nkb : mx;
            }
            CHECK(next == nk && mx - mn <= 1, "nk=%d S=%d split", nk, S);
        }
    }
    // split choice: 1..kMaxSplits, at least 2 k-blocks per split when split,
    // with and without the resident-cluster table (GB300, 152 SMs)
    const int clusters[kMaxSplits + 1] = {0, 456, 228, 148, 110, 87, 74, 59, 51};
    for (int n_tiles = 1; n_tiles <= 512; ++n_tiles)
        for (int nk = 1; nk <= 240; nk += 7)
            for (const int* cl : {static_cast<const int*>(nullptr), clusters}) {
                const int S = choose_splits(n_tiles, nk, 152, cl);
                CHECK(S >= 1 && S <= kMaxSplits, "tiles=%d nk=%d S=%d", n_tiles, nk, S);
                CHECK(S == 1 || nk >= 2 * S, "tiles=%d nk=%d S=%d", n_tiles, nk, S);
            }
    // the 8B decode layers split as measured: 32 slabs of 4096 -> 8, the
    // 224 slabs of 4096 -> 28672 -> 2
    CHECK(choose_splits(32, 32, 152, clusters) == 8, "O-proj split");
    CHECK(choose_splits(224, 32, 152, clusters) == 2, "gate/up split");
    // wide token tiles: the fewest waves, then the largest split (brute force)
    for (int n_tiles = 1; n_tiles <= 400; n_tiles += 3)
        for (int nk = 1; nk <= 120; nk += 5)
            for (int slots : {152, 304})
                for (const int* cl : {static_cast<const int*>(nullptr), clusters}) {
                    const int S = choose_splits_min_waves(n_tiles, nk, slots, cl);
                    auto waves = [&](int s) {
                        const int pw = (cl && cl[s] > 0) ? cl[s] : slots / s;
                        return (n_tiles + pw - 1) / pw;
                    };
                    CHECK(S >= 1 && S <= kMaxSplits && (S == 1 || nk >= 2 * S),
                          "wide tiles=%d nk=%d S=%d", n_tiles, nk, S);
                    for (int s = 1; s <= kMaxSplits && (s == 1 || nk >= 2 * s); ++s) {
                        CHECK(waves(s) >= waves(S), "wide tiles=%d nk=%d: S=%d not fewest", n_tiles,
                              nk, S);
                        CHECK(!(waves(s) == waves(S) && s > S), "wide tiles=%d nk=%d: S=%d not largest",
                              n_tiles, nk, S);
                    }
                }
    // pulled tiles: about 256 CTAs, every cluster resident, >= 2 k-blocks
    for (int n_tiles = 1; n_tiles <= 512; ++n_tiles)
        for (int nk = 1; nk <= 240; nk += 7) {
            const int S = choose_splits_pull(n_tiles, nk, clusters);
            CHECK(S >= 1 && S <= kMaxSplits && (S == 1 || nk >= 2 * S),
                  "pull tiles=%d nk=%d S=%d", n_tiles, nk, S);
            CHECK(S == 1 || clusters[S] >= n_tiles, "pull tiles=%d S=%d not resident", n_tiles, S);
        }
    CHECK(choose_splits_pull(80, 64, clusters) == 3, "70B QKV at 32 tokens");
    CHECK(choose_splits_pull(64, 64, clusters) == 4, "70B O at 32 tokens");
    CHECK(choose_splits_pull(64, 224, clusters) == 4, "70B down at 32 tokens");
    CHECK(choose_splits_pull(448, 64, clusters) == 1, "70B gate/up at 32 tokens");
    CHECK(choose_splits_pull(48, 32, clusters) == 5, "8B QKV at 32 tokens");
    // 224 slabs on 304 slots fit one wave unsplit; 48 slabs take the largest
    // split that still fits one wave
    CHECK(choose_splits_min_waves(224, 32, 304, nullptr) == 1, "wide gate/up");
    CHECK(choose_splits_min_waves(48, 32, 304, nullptr) == 6, "wide QKV");
    std::printf(fails ? "FAIL %d\n" : "OK\n", fails);
    return fails ? 1 : 0;
}
"""


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="needs nvcc (host compile only)")
def test_split_k_host_arithmetic(tmp_path):
    src = tmp_path / "split_host.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "split_host"
    r = subprocess.run(["nvcc", "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip().endswith("OK"), out.stdout[-2000:]
