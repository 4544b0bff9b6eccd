"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/oracle.c``, plants one mistake (a dropped term, a
wrong sign, a wrong operand or index), compiles the copy into a temporary
library and checks that at least one pin -- the padded torch recomputation or
central finite differences -- rejects it.  The mistakes live only in the
temporary copy.
"""
import pytest

import oracle
import workloads
from tests.test_oracle_pins import finite_difference_errors, torch_reference_errors

SRC = oracle.SRC.read_text()

MUTANTS = {
    "delta_sign": ("ds[j] = p[j] * (dp - delta);", "ds[j] = p[j] * (dp + delta);"),
    "delta_dropped": ("ds[j] = p[j] * (dp - delta);", "ds[j] = p[j] * dp;"),
    "dq_scale_dropped": ("dst[d] += scale * ds[j] * kb[j * ld + d];", "dst[d] += ds[j] * kb[j * ld + d];"),
    "dq_scale_dropped_full": ("dq[i * lddq + d] += scale * sij * kj[d];", "dq[i * lddq + d] += sij * kj[d];"),
    "dk_operand": ("dk[j * lddk + d] += scale * sij * qi[d];", "dk[j * lddk + d] += scale * pij * qi[d];"),
    "dv_operand": ("dv[j * lddk + d] += pij * doi[d];", "dv[j * lddk + d] += sij * doi[d];"),
    "lse_max_dropped": ("const double lse = mx + log(sum);", "const double lse = log(sum);"),
    "score_scale_dropped": ("p[j] = scale * dot;", "p[j] = dot;"),
    "p_unnormalised": ("p[j] = exp(p[j] - lse);", "p[j] = exp(p[j] - mx);"),
    "dp_wrong_row": ("dp += doi[d] * vj[d];", "dp += doi[d] * v[d];"),
    "dq_wrong_operand": ("dq[i * lddq + d] += scale * sij * kj[d];",
                         "dq[i * lddq + d] += scale * sij * (v + j * ldk)[d];"),
    "broadcast_offset": ("orow = (int64_t)b * Lq + i;", "orow = i;"),
}


def _mutant(tmp_path, name):
    before, after = MUTANTS[name]
    assert SRC.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / f"{name}.c"
    src.write_text(SRC.replace(before, after))
    lib = oracle.build(src, tmp_path / f"lib{name}.so", force=True)
    return oracle.Oracle(lib)


def _caught(orc) -> bool:
    probs = [
        workloads.make_problem(3, 2, 8, "self", [3, 5, 2], seed=21),
        workloads.make_problem(3, 2, 8, "broadcast", [4, 2, 6], Lq=3, seed=22),
    ]
    for p in probs:
        errs = torch_reference_errors(orc, p)
        if max(errs.values()) > 1e-9:
            return True
        rows = list(range(p.n_q_rows))
        full = orc.bwd(p.q, p.k, p.v, p.dout, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D,
                       p.scale)[0]
        for h in range(p.H):
            got = orc.dq_rows(p.q, p.k, p.v, p.dout, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq,
                              p.D, p.scale, h, rows)
            if (got - full[:, h]).abs().max() > 1e-9:
                return True
    p = workloads.make_problem(2, 1, 4, "self", [3, 2], seed=23)
    return max(finite_difference_errors(orc, p).values()) > 1e-6


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    assert _caught(_mutant(tmp_path, name)), f"no pin caught mutant {name}"


def test_unmutated_oracle_passes_the_same_checks():
    assert not _caught(oracle.default())
