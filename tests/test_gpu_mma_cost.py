"""What a tensor-core product costs on this GPU (jfa_selftest_mma_cycles),
measured from one thread with the loop unrolled and the form fixed at
compile time, to the completion of the final commit:

* issued back to back, an M = 128, K = 16 bf16 product runs at the tensor
  core's rate -- 128 x N x 16 x 2 flops at 8192 flop/cycle/SM, 64 cycles at
  N = 128, 128 at N = 256 -- in SS and TS (A in TMEM) form alike, with K-major
  or MN-major (transposed) shared-memory operands alike, and the issuing
  thread keeps pace with the pipe;
* when each group of eight products must complete before the next group is
  issued (a dependent chain, as in the kernels: a group's results feed the
  work the next one needs) the group costs its eight products plus several
  hundred cycles of latency, so the pipe idles for a large share of the time.

The kernels' per-block and per-step times are read against these two numbers."""
import pytest

import jagged_attention_gb300 as jfa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


def _best(form, group=0):
    runs = [jfa.selftest_mma_cycles(form, 4096, group) for _ in range(3)]
    return min(r[0] for r in runs), min(r[1] for r in runs)


def test_product_cost():
    names = ("M128 N128", "M128 N256", "M128 N128 A-in-TMEM", "M128 N64", "M128 N128 B-MN",
             "M128 N128 A-MN B-MN", "M128 N128 A-in-TMEM B-MN")
    c = {f: _best(f) for f in range(7)}
    g8 = _best(0, 8)
    print("cycles per product (completion / issue): " +
          ", ".join(f"{names[f]} {c[f][0]:.1f} / {c[f][1]:.1f}" for f in range(7)) +
          f"; M128 N128 in dependent groups of 8: {g8[0]:.1f} per product, {8 * g8[0]:.0f} per group")
    n128, n256, ts128, n64 = c[0][0], c[1][0], c[2][0], c[3][0]
    # the math of a 128x128x16 product is 64 cycles at 8192 flop/cycle/SM
    assert 60 <= n128 <= 80
    assert 1.8 * n128 <= n256 <= 2.2 * n128
    assert 0.9 * n128 <= ts128 <= 1.1 * n128
    assert n64 < n128
    # transposed (MN-major) operands cost the same as K-major ones
    for f in (4, 5, 6):
        assert 0.9 * n128 <= c[f][0] <= 1.1 * n128
    assert c[0][1] >= 0.9 * n128            # the issuing thread keeps pace with the pipe
    # a dependent group of eight pays its latency on top of its products
    assert 8 * g8[0] >= 8 * n128 + 200
