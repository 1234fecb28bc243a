"""Host logic of bench.py that needs no GPU: the workload variants (group size, no scales, the
epilogue, device-resident token counts) and their algorithmic byte counts."""
import types

import numpy as np
import pytest

import bench
import wq4_inputs as I


def _args(**kw):
    a = dict(workload="decode_m8_n4096_k4096_bf16_u4b8", group_size=I.GROUP, no_scales=False, epilogue=False,
             device_m=False)
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_plain_workload_is_unchanged():
    """No variant flag: the same seeded inputs, bytes and config as the named workload."""
    for name in I.WORKLOADS:
        a = _args(workload=name)
        assert bench.variant_of(a) == {}
        got, ref = bench.make_inputs(a), I.make_workload(name)
        got = got if isinstance(got, list) else [got]
        ref = ref if isinstance(ref, list) else [ref]
        assert len(got) == len(ref)
        for g, r in zip(got, ref):
            assert (g.M, g.N, g.K, g.qtype, g.dtype) == (r.M, r.N, r.K, r.qtype, r.dtype)
            assert np.array_equal(g.X_bits, r.X_bits) and np.array_equal(g.Wq, r.Wq)
            assert np.array_equal(g.S_bits, r.S_bits)
            assert bench.variant_bytes(g, a) == I.algorithmic_bytes(r.M, r.N, r.K, r.qtype)


def test_variant_bytes():
    """Scales counted as the variant has them; C and bias read once by the epilogue."""
    M, N, K = 8, 4096, 4096
    base = I.algorithmic_bytes(M, N, K, I.U4B8)
    p = bench.make_inputs(_args(group_size=K))
    assert p.S_bits.shape == (1, N)
    assert bench.variant_bytes(p, _args(group_size=K)) == base - 2 * (K // 128 - 1) * N
    p = bench.make_inputs(_args(no_scales=True))
    assert p.S_bits is None
    assert bench.variant_bytes(p, _args(no_scales=True)) == base - 2 * (K // 128) * N
    p = bench.make_inputs(_args(epilogue=True))
    assert bench.variant_bytes(p, _args(epilogue=True)) == base + 2 * M * N + 2 * N
    assert set(bench.variant_of(_args(epilogue=True, group_size=512))) == {"epilogue", "group_size"}


def test_variant_rules():
    with pytest.raises(SystemExit):        # zero points need their scales
        bench.make_inputs(_args(workload="asym_m128_n14336_k4096_bf16_u4zp", no_scales=True))
    with pytest.raises(SystemExit):        # the grouped call has no epilogue
        bench.make_inputs(_args(workload="grouped_8x_n14336_k4096_summ1024_bf16_u4b8", epilogue=True))
    g = bench.make_inputs(_args(workload="grouped_8x_n14336_k4096_summ1024_bf16_u4b8", device_m=True))
    assert isinstance(g, list) and sum(p.M for p in g) == 1024
    a = _args(workload="grouped_8x_n14336_k4096_summ1024_bf16_u4b8", dev_ptrs=True)
    assert bench.variant_of(a) == {"pointers": "device memory (wq4_grouped_mm_dev_ptrs)"}
    assert sum(p.M for p in bench.make_inputs(a)) == 1024


def test_reference_arm_line(capsys):
    """bench.py --impl reference (the oracle on the host cores) prints one JSON line with the keys
    the driver reads, on the default workload's metric and config."""
    import json
    import sys
    argv = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"]
    try:
        bench.main()
    finally:
        sys.argv = argv
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["config"]["workload"] == bench.DEFAULT_WORKLOAD and d["value"] > 0
    assert {"value", "unit", "cores", "kind", "sample"} <= set(d["cpu_baseline"])
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_default_run_covers_every_workload():
    """The default bench run measures every named workload, the decode one as the headline."""
    assert sorted(bench.ALL_WORKLOADS) == sorted(I.WORKLOADS)
    assert bench.DEFAULT_WORKLOAD in bench.ALL_WORKLOADS
    assert bench.REPLAYS >= 5


def test_float_zeros_variant():
    """--float-zeros draws the workload's weight in the float-zero format and counts its zeros."""
    a = _args(workload="asym_m128_n14336_k4096_bf16_u4zp", float_zeros=True)
    p = bench.make_inputs(a)
    assert p.qtype == I.U4_FZP and p.Z.dtype == np.uint16 and p.Z.shape == (p.K // 128, p.N)
    assert bench.variant_of(a)["qtype"].startswith("u4_fzp")
    assert bench.variant_bytes(p, a) == I.algorithmic_bytes(p.M, p.N, p.K, I.U4B8) + 2 * (p.K // 128) * p.N
    g = bench.make_inputs(_args(workload="grouped_8x_n14336_k4096_summ1024_bf16_u4b8", float_zeros=True))
    assert all(q.qtype == I.U4_FZP and q.Z.dtype == np.uint16 for q in g) and sum(q.M for q in g) == 1024
