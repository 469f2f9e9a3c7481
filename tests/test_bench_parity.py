"""The bench's parity block (host logic, CPU only): the cpu_baseline leg's
oracle results compared with a step's outputs.  Outputs that are the oracle's
own results rounded to bf16 pass; one wrong query row fails."""
import dataclasses

import numpy as np
import torch

import bench
import oracle
from attn_fwd_gb300.inputs import WORKLOADS, make_workload_inputs


def _small(name, **kw):
    w = WORKLOADS[name]
    return dataclasses.replace(w, name=w.name + "@small", **kw)


def _outputs_from_oracle(w, t):
    """The oracle's own results, rounded to bf16 as a GPU step stores them."""
    bm = t.get("block_mask")
    f = {n: t[n].double().numpy() for n in ("q", "k", "v", "do")}
    o, lse = oracle.forward(f["q"], f["k"], f["v"], w.scale, causal=w.causal,
                            block_mask=None if bm is None else bm.numpy())
    dq, dk, dv, _ = oracle.backward(f["q"], f["k"], f["v"], f["do"], w.scale, causal=w.causal,
                                    block_mask=None if bm is None else bm.numpy())
    bf = lambda x: torch.from_numpy(x).to(torch.bfloat16)
    return {"o": bf(o), "lse": torch.from_numpy(lse).float(), "dq": bf(dq), "dk": bf(dk), "dv": bf(dv)}


def test_parity_block_passes_rounded_oracle_and_catches_a_wrong_row():
    for w in (_small("fwdbwd_b2h16n4096d128_causal", B=1, H=3, N=384),
              _small("fwdbwd_b1h16n8192d128_blocksparse", H=2, N=512)):
        t = make_workload_inputs(w)
        gpu = _outputs_from_oracle(w, t)
        par = bench.Parity()
        _, _, heads = bench._oracle_sample(w, t, budget_s=60.0, gpu=gpu, parity=par)
        rep = par.report(True)
        assert heads == w.B * w.H and rep["heads_checked"] == heads
        assert rep["ok"], rep
        assert rep["grad_element_heads"] == 2 and rep["grad_element_excess"] <= 0
        assert rep["o_excess"] <= 0 and rep["lse_rel"] <= 1e-3
        for name in ("dq", "dk", "dv"):
            bad = {k: v.clone() for k, v in gpu.items()}
            bad[name][0, 0, [130, 131]] = bad[name][0, 0, [131, 130]]
            par = bench.Parity()
            bench._oracle_sample(w, t, budget_s=60.0, gpu=bad, parity=par)
            assert not par.report(True)["ok"], name
        bad = {k: v.clone() for k, v in gpu.items()}
        bad["o"][0, 0, 5] += 0.05
        par = bench.Parity()
        bench._oracle_sample(w, t, budget_s=60.0, gpu=bad, parity=par)
        assert not par.report(True)["ok"]


def test_parity_block_forward_only():
    w = _small("fwd_b1h32n16384d128_causal_x3", H=2, N=640)
    t = make_workload_inputs(w)
    f = {n: t[n].double().numpy() for n in ("q", "k", "v")}
    o, lse = oracle.forward(f["q"], f["k"], f["v"], w.scale, causal=True)
    gpu = {"o": torch.from_numpy(o).to(torch.bfloat16), "lse": torch.from_numpy(lse).float()}
    par = bench.Parity()
    bench._oracle_sample(w, t, budget_s=60.0, gpu=gpu, parity=par)
    rep = par.report(False)
    assert rep["ok"] and rep["heads_checked"] == 2
    gpu["lse"][0, 1, 7] += 0.1
    par = bench.Parity()
    bench._oracle_sample(w, t, budget_s=60.0, gpu=gpu, parity=par)
    assert not par.report(False)["ok"]
    assert np.isfinite(rep["o_max_abs"])
