"""Host logic (CPU): the context CTA share beside concurrent generation work
(pkv::context_cta_share in csrc/internal.h, used by the host for exact plans and by the plan
kernel for bucket plans).  The closed form must land on the minimum of its own cost model over
every CTA count, keep every SM when there is no generation work, and give the context kernel
more SMs the more context work there is."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_rope_gb300", "csrc")
SRC = r'''
#include <cstdio>
#include "internal.h"
int main() {
  float tp, u, gk; int hq, hkv, d, s;
  while (std::scanf("%f %f %f %d %d %d %d", &tp, &u, &gk, &hq, &hkv, &d, &s) == 7)
    std::printf("%d\n", pkv::context_cta_share(tp, u, gk, hq, hkv, d, s));
  return 0;
}
'''


@pytest.fixture(scope="module")
def share(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    cuda_inc = "/usr/local/cuda/include"
    if cxx is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    d = tmp_path_factory.mktemp("share")
    src, exe = d / "share.cpp", d / "share"
    src.write_text(SRC)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-I", cuda_inc,
                    str(src), "-o", str(exe)], check=True)

    def run(rows):
        inp = "".join(" ".join(str(x) for x in r) + "\n" for r in rows)
        out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True).stdout
        return [int(x) for x in out.split()]
    return run


def _cost(tp, u, gk, hq, hkv, d, s, n):
    """The model's step time with n context CTAs (float64; the closed form runs in float32)."""
    t_ctx = 1.3 * (tp * 1.45 + u * 1.9) * hq / s
    t_gen = gk * hkv * d * 4.0 / 6.3e6
    if n >= s:
        return t_ctx + t_gen
    m_sat = 2.0 * s / 3.0
    return max(t_ctx * s / n, t_gen * max(1.0, m_sat / (s - n)))


def test_closed_form_is_the_model_minimum(share):
    rng = np.random.default_rng(5)
    rows = []
    for _ in range(3000):
        s = int(rng.choice([132, 148, 152, 160]))
        rows.append((int(rng.integers(1, 300000)), int(rng.integers(1, 4000)), int(rng.integers(1, 8_000_000)),
                     int(rng.choice([8, 32, 64])), int(rng.choice([1, 8])), int(rng.choice([64, 128])), s))
    got = share(rows)
    for r, n in zip(rows, got):
        s = r[-1]
        assert s // 8 <= n <= s
        best = min(_cost(*r, k) for k in list(range(s // 8, s)) + [s])
        assert _cost(*r, n) <= best * (1 + 1e-5), (r, n)


def test_no_generation_work_keeps_every_sm(share):
    assert share([(5000, 100, 0, 32, 8, 128, 152), (1, 1, 0, 8, 1, 64, 148)]) == [152, 148]


def test_more_context_work_more_ctas(share):
    rows = [(tp, tp // 10, 300_000, 32, 8, 128, 152) for tp in (500, 2000, 8000, 32000, 128000)]
    got = share(rows)
    assert got == sorted(got) and got[0] < got[-1]
