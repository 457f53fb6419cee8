"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

* The five workloads' smaller variants (several chunks, ragged tails, an empty
  sequence) are compared element by element over whole tensors.
* The five full-size workloads run in the launch configuration the benchmark
  times; the oracle recomputes sampled (sequence, head) units one by one.
"""
import pytest
import torch

from gated_delta_rule_36_gb300.inputs import FULL_WORKLOADS, SMALL_WORKLOADS, make_inputs, workload

from kda_testutil import check_full, check_units, oracle_full, oracle_units, run_gpu, seq_bounds

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", SMALL_WORKLOADS)
def test_small_workloads_whole_tensor(name):
    inp = make_inputs(name, "cpu")
    out, final, bits = run_gpu(inp)
    assert bits == 0
    ref_out, ref_final = oracle_full(inp)
    check_full(inp, out, final, ref_out, ref_final)


def _sample_units(w, gen):
    bounds = seq_bounds(w)
    lens = [e - b for b, e in bounds]
    order = sorted(range(len(lens)), key=lambda n: (-lens[n], n))
    seqs = {order[0], order[-1]} | {int(x) for x in torch.randint(0, len(lens), (2,), generator=gen)}
    units = set()
    for n in seqs:
        units.add((n, 0))
        units.add((n, w.H - 1))
        units.add((n, int(torch.randint(0, w.H, (1,), generator=gen))))
    return sorted(units)


@pytest.mark.parametrize("name", FULL_WORKLOADS)
def test_full_workloads_sampled_units(name):
    w = workload(name)
    inp = make_inputs(w, "cuda" if name in ("long", "packed64") else "cpu")
    out, final, bits = run_gpu(inp)
    assert bits == 0
    gen = torch.Generator().manual_seed(7)
    units = _sample_units(w, gen)
    if name == "long":
        units = [(0, 0), (0, w.H - 1)]
    ref = oracle_units(inp, units)
    check_units(inp, out, final, ref)
    # bit-exact indexing: rows outside every sequence stay untouched
    last = seq_bounds(w)[-1][1]
    assert torch.isnan(out.reshape(w.B * w.T, w.H, w.V)[last:].float()).all()
    assert torch.isfinite(out.float()).all() if last == w.B * w.T else True
