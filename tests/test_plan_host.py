"""The host-side plan choice (plan.h), compiled with the host compiler and run
on the CPU: decode shapes pack the query heads of a KV head into one tile and
split the keys; prefill shapes use one head per tile and split only when the
grid would leave most SMs idle."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r'''
#include <stdio.h>
#include "exact_tiled_attention_online_gb300/csrc/plan.h"
using namespace attn;
int main() {
  int b, mq, mk, hq, hkv, sms, w;
  while (scanf("%d %d %d %d %d %d %d", &b, &mq, &mk, &hq, &hkv, &sms, &w) == 7) {
    TcPlan p = choose_fwd_plan(b, mq, mk, b * mq, hq, hkv, 128, w, ATTN_DTYPE_BF16, sms);
    printf("%d %d %d %d\n", p.kind, p.pack, p.tile_tokens, p.n_splits);
  }
}
'''


@pytest.fixture(scope="module")
def plan_bin(tmp_path_factory):
    if not shutil.which("g++"):
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("plan")
    src, exe = d / "plan.cpp", d / "plan"
    src.write_text(SRC)
    subprocess.run(["g++", "-std=c++17", "-DATTN_TC_FWD=1", f"-I{ROOT}", "-o", str(exe), str(src)],
                   check=True)
    return str(exe)


def plan(exe, *shape, window=0):
    out = subprocess.run([exe], input=" ".join(map(str, shape + (window,))), capture_output=True,
                         text=True, check=True).stdout.split()
    return tuple(int(x) for x in out)


def test_decode_packs_and_splits(plan_bin):
    kind, pack, tokens, splits = plan(plan_bin, 32, 1, 32768, 32, 8, 152)
    assert (kind, pack, tokens) == (2, 1, 32) and splits >= 2
    kind, pack, tokens, splits = plan(plan_bin, 32, 16, 32768, 32, 8, 152)
    assert (kind, pack, tokens) == (2, 1, 32) and splits >= 2


def test_prefill_one_head_per_tile_no_split(plan_bin):
    for shape in ((4, 4096, 4096, 32, 8), (1, 1024, 1024, 32, 8), (2, 8192, 8192, 16, 4)):
        assert plan(plan_bin, *shape, 152) == (1, 0, 128, 1), shape


def test_long_single_query_mha_splits(plan_bin):
    kind, pack, tokens, splits = plan(plan_bin, 1, 1, 100000, 32, 32, 152)
    assert kind == 2 and pack == 0 and splits > 1


def test_short_window_decode_does_not_split(plan_bin):
    """A bounded window of 512 keys leaves a decode tile six key tiles, too few
    to split; a long window still splits like the unbounded decode."""
    assert plan(plan_bin, 32, 1, 32768, 32, 8, 152, window=512) == (1, 1, 32, 1)
    kind, pack, tokens, splits = plan(plan_bin, 32, 1, 32768, 32, 8, 152, window=8192)
    assert (kind, pack) == (2, 1) and splits >= 2


def test_empty_query_batch_plans_without_split(plan_bin):
    """No query rows (max_seqlen_q = 0, or batch = 0) is a legal no-op: the
    planner returns a plan without a key split instead of dividing by its
    zero CTA count ("causal-mask-and-ragged-sequence-layouts", fifth
    paragraph: empty batches where the API permits them)."""
    for shape in ((2, 0, 4096, 32, 8), (2, 0, 32768, 32, 8), (1, 0, 100000, 32, 32),
                  (0, 0, 32768, 32, 8), (0, 16, 32768, 32, 8)):
        kind, pack, tokens, splits = plan(plan_bin, *shape, 152)
        assert kind == 1 and splits == 1, shape
    assert plan(plan_bin, 2, 0, 32768, 32, 8, 152, window=4096)[3] == 1


def test_fp32_takes_cuda_cores(plan_bin, tmp_path):
    src = SRC.replace("ATTN_DTYPE_BF16", "ATTN_DTYPE_FP32")
    (tmp_path / "p.cpp").write_text(src)
    subprocess.run(["g++", "-std=c++17", "-DATTN_TC_FWD=1", f"-I{ROOT}", "-o",
                    str(tmp_path / "p"), str(tmp_path / "p.cpp")], check=True)
    assert plan(str(tmp_path / "p"), 4, 4096, 4096, 32, 8, 152)[0] == 0
