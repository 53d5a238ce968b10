"""Host logic of bench.py, without a GPU.

The bench runs its GPU reports only on a GPU, where a slip in their Python would cost the
whole line; these tests drive the reporting functions through stand-ins for the CUDA
calls (events, graphs and the library's entry points) to check their shapes, the buffers
they hand to the library and the JSON they produce.  The reference arm (the CPU oracle)
runs for real on a small sample.
"""

import contextlib
import io
import json
import os
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import gemm_cq_gemv_gb300 as cqlib  # noqa: E402
from gemm_cq_gemv_gb300 import synth  # noqa: E402


class _Event:
    def __init__(self, enable_timing=True):
        pass

    def record(self, *a):
        pass

    def elapsed_time(self, other):
        return 0.25


class _Graph:
    def __init__(self):
        self.fn = None

    def replay(self):
        self.fn()


def _fake_torch():
    @contextlib.contextmanager
    def graph(g, stream=None):
        yield

    cuda = types.SimpleNamespace(
        Event=_Event, synchronize=lambda: None, empty_cache=lambda: None,
        Stream=lambda *a, **k: types.SimpleNamespace(wait_stream=lambda o: None),
        current_stream=lambda: None, CUDAGraph=_Graph, graph=graph,
        get_device_properties=lambda d: types.SimpleNamespace(L2_cache_size=4 << 20))
    ft = types.SimpleNamespace(**{k: getattr(torch, k) for k in
                                  ("empty", "uint8", "float32", "randn", "Generator", "int8", "int16")})
    ft.cuda = cuda
    return ft


class _FakeLib:
    """Stand-in for the library's entry points: checks what the bench hands over."""

    CQ_TERNARY = cqlib.CQ_TERNARY
    cq_gemv_workspace_bytes = staticmethod(cqlib.cq_gemv_workspace_bytes)

    def __init__(self):
        self.calls = {}

    def _count(self, name):
        self.calls[name] = self.calls.get(name, 0) + 1

    @staticmethod
    def _ok(t):
        assert t.is_contiguous() and t.data_ptr() % 16 == 0

    def cq_encode(self, W, b, cb):
        N, K = W.shape
        f = cqlib.cq_field_bits(b)
        return (torch.zeros((N, K // 128, 16 * f), dtype=torch.uint8),
                torch.zeros((N, K // 128), dtype=torch.int16))

    def a8_quantize(self, X, Xq=None, scale=None):
        self._count("a8_quantize")
        return torch.zeros(X.shape, dtype=torch.int8), torch.ones(X.shape[0])

    LAYER_MAX_PROBLEMS = cqlib.LAYER_MAX_PROBLEMS

    def make_gemv_layer(self, items):
        for packed, norms, N, K, X, Y in items:
            self._ok(packed), self._ok(norms)
            assert packed.shape == (N, K // 128, 64) and X.shape == (1, K) and Y.shape == (1, N)
        assert len(items) <= self.LAYER_MAX_PROBLEMS
        return list(items)

    def make_q4_0_layer(self, items):
        for blocks, N, K, X, Y in items:
            self._ok(blocks)
            assert blocks.shape == (N, -(-K // 32) * 18) and X.shape == (1, K) and Y.shape == (1, N)
        assert len(items) <= self.LAYER_MAX_PROBLEMS
        return list(items)

    def cq_gemv_layer(self, probs, b, cb):
        self._count("cq_gemv_layer")
        self.calls["cq_layer_problems"] = self.calls.get("cq_layer_problems", 0) + len(probs)

    def q4_0_gemv_layer(self, probs):
        self._count("q4_0_gemv_layer")
        assert len(probs) == 8

    def cq_gemv(self, packed, norms, N, K, b, cb, Xq, s, Y=None, workspace=None):
        self._ok(packed), self._ok(norms)
        assert packed.shape == (N, K // 128, 16 * cqlib.cq_field_bits(b))
        assert Y.shape == (Xq.shape[0], N)
        Y.fill_(1.0)
        self._count("cq_gemv")

    def cq_gemv_lut(self, packed, norms, N, K, b, cb, Xq, s, Y=None):
        self._ok(packed), self._ok(norms)
        assert b in (1, 2, cqlib.CQ_TERNARY)
        Y.fill_(1.0)
        self._count("cq_gemv_lut")

    def q4_0_quantize(self, W):
        N, K = W.shape
        return torch.zeros((N, -(-K // 32) * 18), dtype=torch.uint8)

    def q4_0_gemv(self, blocks, N, K, X, Y=None):
        self._ok(blocks)
        assert blocks.shape == (N, -(-K // 32) * 18) and X.shape[1] == K
        self._count("q4_0_gemv")

    def q4_0_gemm_workspace_bytes(self, M, K):
        return M * (-(-K // 32) * 32) * 2

    def q4_0_gemm(self, blocks, N, K, X, Y=None, workspace=None):
        self._ok(blocks), self._ok(workspace)
        assert Y.shape == (X.shape[0], N) and workspace.numel() >= self.q4_0_gemm_workspace_bytes(*X.shape)
        self._count("q4_0_gemm")

    def cq_device_error(self):
        pass


def test_small_report_shapes_and_copies(monkeypatch):
    def capture(torch_, fn):
        g = _Graph()
        g.fn = fn
        fn()
        return g

    monkeypatch.setattr(bench, "_capture", capture)
    lib = _FakeLib()
    out = bench.small_report("cpu", None, _fake_torch(), lib, synth, 2, 1)
    a, b = out["cq_w4a8_512x512"], out["minueza_q4_0_layer"]
    assert a["bytes_per_call"] == 512 * 512 // 2 + 2 * 512 * 4 + 4 * 512 + 4 * 512
    assert a["copies"] * a["bytes_per_call"] >= 4 * out["l2_bytes"]
    assert a["launches"] == 1 and b["launches"] == 1 and b["unfused_launches"] == 8
    assert b["copies"] * b["bytes_per_layer"] >= 4 * out["l2_bytes"]
    assert b["bytes_per_layer"] >= 6_499_800            # the layer's Q4_0 blocks alone
    # latency: capture + (warmup + steps) replays; streamed: capture + 1 + 3 replays, once
    # with one call per copy and once with 16 copies per call
    n16 = -(-a["copies"] // lib.LAYER_MAX_PROBLEMS)
    assert out["launch_floor_us"] > 0
    assert lib.calls["cq_gemv_layer"] == 1 + 3 + (1 + 1 + 3) * (a["copies"] + n16)
    assert lib.calls["cq_layer_problems"] == 1 + 3 + (1 + 1 + 3) * 2 * a["copies"]
    assert lib.calls["cq_gemv"] == lib.calls["a8_quantize"] == 1 + 3     # the unfused latency
    assert lib.calls["q4_0_gemv_layer"] == 1 + 3 + (1 + 1 + 3) * b["copies"]
    assert lib.calls["q4_0_gemv"] == 8 * (1 + 3)
    json.dumps(out)


def test_narrow_report_covers_every_code_and_shape():
    lib = _FakeLib()
    small = tuple(types.SimpleNamespace(name=m.name, N=m.N // 128, K=m.K) for m in synth.LARGE)
    fs = types.SimpleNamespace(LARGE=small, weight_seed=synth.weight_seed,
                               activation_seed=synth.activation_seed)
    out = bench.narrow_report("cpu", None, _fake_torch(), lib, fs, 2, 3)
    for key in ("b1", "b2", "ternary"):
        assert set(out[key]["cq_gemv"]["us"]) == {m.name for m in small}
        assert out[key]["cq_gemv_lut"]["GBps"] > 0
        assert out[key]["max_rel_diff"] == 0.0
    assert lib.calls["cq_gemv"] == lib.calls["cq_gemv_lut"] == 3 * 4 * (3 + 2)
    json.dumps(out)


def test_reference_arm_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-rows", "4"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--steps", "1", "--warmup", "2"])


def test_blas_thread_count(monkeypatch):
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        monkeypatch.delenv(v, raising=False)
    assert bench.blas_threads() == os.cpu_count()
    monkeypatch.setenv("OMP_NUM_THREADS", "1")
    assert bench.blas_threads() == 1


def test_cpu_baseline_only_entry(monkeypatch):
    """The one-thread child of a full run prints exactly the oracle timing as JSON."""
    monkeypatch.setattr(bench, "cpu_baseline", lambda rows: {"value": 1.0, "rows": rows})
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--cpu-baseline-only", "--cpu-rows", "3"])
    assert json.loads(buf.getvalue()) == {"value": 1.0, "rows": 3}


def test_batched_report_shapes():
    lib = _FakeLib()
    ft = _fake_torch()
    small = tuple(types.SimpleNamespace(name=m.name, N=m.N // 256, K=m.K) for m in synth.LARGE)
    mats = []
    for m in small:
        W = torch.zeros((m.N, m.K))
        packed, norms = lib.cq_encode(W, 4, None)
        mats.append(dict(m=m, packed=packed, norms=norms, blocks=lib.q4_0_quantize(W)))
    out = bench.batched_report(mats, None, ft, lib, synth, "cpu", 2, 1, batches=(8, 32))
    for B in (8, 32):
        assert set(out[f"B{B}"]) == {"cq_gemv", "q4_0_gemm"}
        assert set(out[f"B{B}"]["cq_gemv"]["us"]) == {m.name for m in small}
    assert lib.calls["cq_gemv"] == lib.calls["q4_0_gemm"] == 2 * 4 * (1 + 2)
    json.dumps(out)


def test_batched_report_batch_two_uses_the_gemvs():
    lib = _FakeLib()
    ft = _fake_torch()
    small = tuple(types.SimpleNamespace(name=m.name, N=m.N // 256, K=m.K) for m in synth.LARGE)
    mats = []
    for m in small:
        W = torch.zeros((m.N, m.K))
        packed, norms = lib.cq_encode(W, 4, None)
        mats.append(dict(m=m, packed=packed, norms=norms, blocks=lib.q4_0_quantize(W)))
    out = bench.batched_report(mats, None, ft, lib, synth, "cpu", 2, 1, batches=(2,), hbm=1000.0)
    assert set(out["B2"]) == {"cq_gemv", "q4_0_gemv"}
    assert out["B2"]["q4_0_gemv"]["frac_of_hbm"] > 0
    assert "q4_0_gemm" not in lib.calls and lib.calls["q4_0_gemv"] == 4 * (1 + 2)


def test_mixed_report_covers_every_width_shape_and_batch(monkeypatch):
    def capture(torch_, fn):
        g = _Graph()
        g.fn = fn
        fn()
        return g

    monkeypatch.setattr(bench, "_capture", capture)
    lib = _FakeLib()
    small = tuple(types.SimpleNamespace(name=m.name, N=m.N // 64, K=m.K // 8) for m in synth.CQ_MIXED)
    fs = types.SimpleNamespace(CQ_MIXED=small, CQ_MIXED_BITS=synth.CQ_MIXED_BITS,
                               CQ_MIXED_BATCHES=synth.CQ_MIXED_BATCHES,
                               weight_seed=synth.weight_seed, activation_seed=synth.activation_seed)
    ft = _fake_torch()
    ft.rand = torch.rand
    ft.where = torch.where
    out = bench.mixed_report("cpu", None, ft, lib, fs, 2, 3, 1e-3)
    l2 = 4 << 20                                   # the fake device's L2
    calls = 0
    for m in small:
        for b in (1, 2, 3, 4):
            wbytes = m.N * (m.K // 128) * 16 * cqlib.cq_field_bits(b) + 2 * m.N * (m.K // 128)
            copies = -(-4 * l2 // wbytes)          # distinct copies spanning 4x the L2
            for B in (1, 4, 16):
                k = f"{m.name}_b{b}_B{B}"
                assert out[k + "_us"] > 0 and out[k + "_frac"] > 0 and out[k + "_Gwps"] > 0
                assert out[k + "_streamed_us"] > 0 and out[k + "_streamed_frac"] > 0
                # flushed: warmup + steps; streamed: capture + 1 + 3 replays of every copy
                calls += (3 + 2) + (1 + 1 + 3) * copies
    assert lib.calls["cq_gemv"] == calls
    json.dumps(out)


def test_summary_flattens_every_workload():
    line = {"small": {"cq_w4a8_512x512": {"latency_us": 5.0, "streamed_GBps": 100.0},
                      "minueza_q4_0_layer": {"latency_us": 20.0, "streamed_GBps": 200.0}},
            "mixed": {"sq_b4_B1_frac": 0.5, "sq_b4_B1_us": 3.0},
            "prefill": {"M512_tflops": 700.0, "M512_frac": 0.36, "M2048_tflops": 1000.0,
                        "M2048_frac": 0.52},
            "kernels": {"cq_gemv": {"GBps": 500.0}},
            "batched": {"B2": {"cq_gemv": {"GBps": 400.0}}, "workload": "x"},
            "cpu_baseline": {"parity": {"ok": True, "cq_gemv_max_rel_err": 1e-7,
                                        "q4_0_gemv_max_rel_err": 2e-6}}}
    s = bench.summary_of(line, 1000.0)
    assert s["cq512_streamed_frac"] == 0.1 and s["minueza_q4_0_layer_latency_us"] == 20.0
    assert s["mixed_sq_b4_B1_frac"] == 0.5 and "mixed_sq_b4_B1_us" not in s
    assert s["prefill_M2048_frac"] == 0.52 and s["decode_B1_cq_gemv_frac"] == 0.5
    assert s["decode_B2_cq_gemv_frac"] == 0.4 and s["oracle_check_ok"] is True
    assert all(not isinstance(v, dict) for v in s.values())


def test_cpu_baseline_checks_a_gpu_sample():
    """The oracle leg run on sampled rows of the step, with the GPU outputs replaced by the
    oracle's own (ok) and by a perturbed copy (not ok)."""
    import numpy as np
    import oracle
    from tests.util import fitted_cb28
    rows = 4
    state = bench.oracle_state(rows, fitted_cb28(), synth, oracle)
    outs = []
    bench.oracle_sample_step(rows, fitted_cb28(), synth, oracle, state, outs)
    sample = [dict(d, y_cq=o[0].astype(np.float32), y_q4=o[1].astype(np.float32))
              for d, o in zip(state, outs)]
    r = bench.cpu_baseline(rows, seconds=0.01, sample=sample)
    assert r["parity"]["ok"] and r["parity"]["cq_gemv_max_rel_err"] < 1e-6
    sample[0]["y_q4"] = sample[0]["y_q4"] * 1.01
    r = bench.cpu_baseline(rows, seconds=0.01, sample=sample)
    assert not r["parity"]["ok"] and r["parity"]["q4_0_gemv_max_rel_err"] > 5e-3
