"""The tile planner and per-lane mask predicates of common.cuh, compiled for
the host with nvcc and run on the CPU, against the oracle's materialised mask
("causal-mask-and-ragged-sequence-layouts", first to fourth paragraphs;
bounded windows: "attention-algorithm-error-and-complexity-tests", fifth
paragraph).

Three views of the same rule must each equal the oracle bit for bit:
  * forward tiles: a tile of query rows visits key blocks [n_begin, n_end)
    (128 keys, or 64 in the two-tile prefill),
    treats the planner's full tiles as allowed without a test, and applies
    the per-row interval test on the others;
  * backward dK/dV tiles: a 128-key tile visits 64-row query tiles from
    row_begin(first key) to row_end(last key) and applies the per-key row
    interval test;
  * the two-tile prefill CTA: tile B's key range starts no later than tile
    A's ends, so the CTA's key loop has no unused tile.
This is the host half of the GPU mask probe: it needs no GPU and covers many
more shapes and windows.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r'''
#include <stdio.h>
#include <vector>
#include "exact_tiled_attention_online_gb300/csrc/common.cuh"
#include "exact_tiled_attention_online_gb300/csrc/plan.h"
using namespace attn;
// stdin: batch mask window tile_rows key_block, then batch pairs (nq nk)
// stdout: forward-view matrix, backward-view matrix (one row per line),
//         then "contiguous <0|1>" and "oob <count>"
int main() {
  int batch, mask, window, tr, bn;
  if (scanf("%d %d %d %d %d", &batch, &mask, &window, &tr, &bn) != 5) return 1;
  std::vector<int> nq(batch), nk(batch), cq(batch + 1, 0), ck(batch + 1, 0);
  for (int s = 0; s < batch; s++) {
    if (scanf("%d %d", &nq[s], &nk[s]) != 2) return 1;
    cq[s + 1] = cq[s] + nq[s];
    ck[s + 1] = ck[s] + nk[s];
  }
  const int TQ = cq[batch], TK = ck[batch];
  std::vector<char> fw((size_t)TQ * TK, '0'), bw((size_t)TQ * TK, '0');
  int contiguous = 1, oob = 0;
  for (int s = 0; s < batch; s++) {
    const int q = nq[s], k = nk[s];
    for (int i0 = 0; i0 < q; i0 += tr) {  // forward view
      const KvRange kr = plan_kv_tiles(mask, window, q, k, i0, tr, bn);
      for (int r = 0; r < tr; r++) {
        const int i = i0 + r;
        if (i >= q) continue;
        for (int n = kr.n_begin; n < kr.n_end; n++)
          for (int c = 0; c < bn; c++) {
            const int j = n * bn + c;
            const bool ok = kr.full(n) || lane_allowed(mask, window, i, j, q, k);
            if (!ok) continue;
            if (j >= k) { oob++; continue; }
            fw[(size_t)(cq[s] + i) * TK + ck[s] + j] = '1';
          }
      }
    }
    for (int i0 = 0; i0 < q; i0 += 2 * kTileRows) {  // two-tile CTA
      const KvRange a = plan_kv_tiles(mask, window, q, k, i0, kTileRows, bn);
      const KvRange b = plan_kv_tiles(mask, window, q, k, i0 + kTileRows, kTileRows, bn);
      if (a.n_end > a.n_begin && b.n_end > b.n_begin &&
          (b.n_begin > a.n_end || b.n_begin < a.n_begin || b.n_end < a.n_end))
        contiguous = 0;
    }
    for (int j0 = 0; j0 < k; j0 += 128) {  // backward dK/dV view, 64-row steps
      const int j_last = (j0 + 128 < k ? j0 + 128 : k) - 1;
      const int m_begin = row_begin(mask, j0, q, k) / 64;
      const int m_end = (row_end(mask, window, j_last, q, k) + 63) / 64;
      for (int m = m_begin; m < m_end; m++)
        for (int c = 0; c < 64; c++) {
          const int i = m * 64 + c;
          for (int r = 0; r < 128; r++) {
            const int j = j0 + r;
            const int rb = key_row_begin(mask, j, q, k), re = key_row_end(mask, window, j, q, k);
            if (i < rb || i >= re) continue;
            if (i >= q || j >= k) { oob++; continue; }
            bw[(size_t)(cq[s] + i) * TK + ck[s] + j] = '1';
          }
        }
    }
  }
  for (int t = 0; t < TQ; t++) printf("%.*s\n", TK, &fw[(size_t)t * TK]);
  for (int t = 0; t < TQ; t++) printf("%.*s\n", TK, &bw[(size_t)t * TK]);
  printf("contiguous %d\noob %d\n", contiguous, oob);
  return 0;
}
'''


@pytest.fixture(scope="module")
def planner(tmp_path_factory):
    if not shutil.which("nvcc"):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("planner")
    src, exe = d / "planner.cu", d / "planner"
    src.write_text(SRC)
    subprocess.run(["nvcc", "-std=c++17", "-O1", f"-I{ROOT}", "-o", str(exe), str(src)],
                   check=True, capture_output=True, text=True)
    return str(exe)


def run_planner(exe, lq, lk, mask, window, tile_rows, key_block=128):
    text = f"{len(lq)} {mask} {window} {tile_rows} {key_block}\n" + "\n".join(
        f"{a} {b}" for a, b in zip(lq, lk)) + "\n"
    out = subprocess.run([exe], input=text, capture_output=True, text=True,
                         check=True).stdout.split("\n")
    tq, tk = sum(lq), sum(lk)

    def mat(lines):
        if tk == 0:
            return np.zeros((tq, 0), np.uint8)
        return np.array([[c == "1" for c in ln] for ln in lines], np.uint8).reshape(tq, tk)

    fw = mat(out[:tq])
    bw = mat(out[tq:2 * tq])
    tail = dict(ln.split() for ln in out[2 * tq:] if ln.strip())
    return fw, bw, int(tail["contiguous"]), int(tail["oob"])


SHAPES = [
    ((300,), (300,)),
    ((1, 129, 700), (1, 129, 700)),
    ((5, 260), (600, 40)),          # Nq < Nk and Nq > Nk (empty rows)
    ((513, 0, 257), (200, 0, 513)),
    ((1,) * 3, (1000, 129, 128)),   # decode
]
WINDOWS = [0, 1, 2, 64, 127, 128, 129, 300]


@pytest.mark.parametrize("lq,lk", SHAPES, ids=[f"s{i}" for i in range(len(SHAPES))])
@pytest.mark.parametrize("mask", [pins.NONE, pins.TOP_LEFT, pins.BOTTOM_RIGHT])
def test_planner_matches_oracle(planner, lq, lk, mask):
    for window in WINDOWS if mask != pins.NONE else [0]:
        ref = oracle.mask(pins.cu(lq), pins.cu(lk), sum(lq), sum(lk), mask, window)
        for tile_rows, key_block in ((128, 128), (32, 128), (128, 64)):
            fw, bw, contiguous, oob = run_planner(planner, lq, lk, mask, window, tile_rows,
                                                  key_block)
            tag = (mask, window, tile_rows, key_block)
            assert oob == 0, tag
            assert np.array_equal(fw, ref), tag
            assert np.array_equal(bw, ref), tag
            assert contiguous == 1, tag
