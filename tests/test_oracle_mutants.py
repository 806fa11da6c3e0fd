"""The pins must catch plausible mistakes in the oracle.  Each case here copies the oracle's C
source, plants one mistake (a wrong mask, index, sign or operand, a dropped term), builds it
on the CPU and runs the pin suite against it: at least one pin must fail."""
import os

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, text in the source, replacement, occurrence to replace: None = all)
MUTANTS = [
    ("causal mask includes the diagonal", "if (p->causal && j > i)", "if (p->causal && j >= i)", None),
    ("causal mask reversed", "if (p->causal && j > i)", "if (p->causal && j < i)", None),
    ("GQA heads strided, not grouped", "int G = Hq / Hkv, g = h / G;", "int G = Hq / Hkv, g = h % Hkv;", None),
    ("LSE drops the max", "*lse_i = m + log(l);", "*lse_i = log(l);", None),
    ("softmax not normalised", "p_row[j] = exp(s_row[j] - m) / l;", "p_row[j] = exp(s_row[j] - m);", None),
    ("backward drops D", "double ds = p_row[j] * (s_row[j] - Dv);", "double ds = p_row[j] * s_row[j];", None),
    ("dS sign flipped in key pass", "double ds = pij * (dp - Dvec[(long)i * D_stride]);",
     "double ds = pij * (Dvec[(long)i * D_stride] - dp);", None),
    ("dK misses the scale", "dk_j[c] += p->sc * ds * qi[c];", "dk_j[c] += ds * qi[c];", None),
    ("dV uses Q instead of dO", "dv_j[c] += pij * doi[c];", "dv_j[c] += pij * qi[c];", None),
    ("dQ uses V instead of K", "const double *kj = p->k + (long)j * p->kv_stride;\n                for",
     "const double *kj = p->v + (long)j * p->kv_stride;\n                for", None),
    ("varlen K read from the V slot", "p.k = qkv + (long)start * tok + 1L * H * d", "p.k = qkv + (long)start * tok + 2L * H * d", None),
    ("kvcache causal mask top-left aligned", "int last = causal ? L - Nq + i : L - 1;",
     "int last = causal ? i : L - 1;", None),
    ("kvcache causal mask one key late", "int last = causal ? L - Nq + i : L - 1;",
     "int last = causal ? L - Nq + i + 1 : L - 1;", None),
    ("kvcache ignores the cache length", "int L = lens ? lens[b] : Nk;", "int L = Nk;", None),
    ("kvcache GQA heads strided", "kvh = h / G;", "kvh = h % Hkv;", None),
    ("kvcache empty row LSE 0", "if (lse) lse[r] = -INFINITY;", "if (lse) lse[r] = 0.0;", None),
    ("cross bwd causal mask top-left aligned", "int last = causal ? Nk - Nq + i : Nk - 1;",
     "int last = causal ? i : Nk - 1;", None),
    ("cross bwd drops D", "dSi[j] = Pi[j] * (dSi[j] - Dv);", "dSi[j] = Pi[j] * dSi[j];", None),
    ("cross bwd dK misses the scale", "dkb[(long)j * d + c] += sc * dsij * qb[(long)i * d + c];",
     "dkb[(long)j * d + c] += dsij * qb[(long)i * d + c];", None),
    ("cross bwd dV from Q", "dvb[(long)j * d + c] += pij * dob[(long)i * d + c];",
     "dvb[(long)j * d + c] += pij * qb[(long)i * d + c];", None),
    ("default scale is 1/d", "return scale == 0.0 ? 1.0 / sqrt((double)d) : scale;",
     "return scale == 0.0 ? 1.0 / (double)d : scale;", None),
]


def _all_pins():
    calls = []
    for name in dir(pins):
        if not name.startswith("test_") or name == "test_flop_count_matches_page_example":
            continue
        fn = getattr(pins, name)
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        combos = [{}]
        for m in params:
            argnames = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) else m.args[0]
            new = []
            for c in combos:
                for val in m.args[1]:
                    vals = val if len(argnames) > 1 else (val,)
                    nc = dict(c)
                    nc.update(zip(argnames, vals))
                    new.append(nc)
            combos = new
        for c in combos:
            calls.append((name, fn, c))
    return calls


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mutant, tmp_path):
    name, old, new, _ = mutant
    src = open(SRC).read()
    assert old in src, f"mutation site not found: {name}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    lib = oracle.load_library(so)
    caught = []
    for pname, fn, kwargs in _all_pins():
        try:
            fn(lib=lib, **kwargs)
        except Exception:  # an assertion, a NaN comparison, a rejected argument ...
            caught.append(pname)
    assert caught, f"no pin catches: {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    so = oracle.compile_source(SRC, str(tmp_path / "libcopy.so"))
    lib = oracle.load_library(so)
    for pname, fn, kwargs in _all_pins():
        fn(lib=lib, **kwargs)
