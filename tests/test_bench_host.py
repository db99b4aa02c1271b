"""Host-side pieces of bench.py that need no GPU: the clock record keeps only
samples taken inside the timed region and decodes the clock-event reason bits,
and the sampler falls back to nvidia-smi when NVML cannot be loaded."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeLib:
    def __init__(self):
        self.shutdown = 0

    def nvmlShutdown(self):
        self.shutdown += 1
        return 0


class _FakeThread:
    def join(self, timeout=None):
        pass


def _sampler(samples, window):
    s = object.__new__(bench.NvmlClockSampler)
    s.lib = _FakeLib()
    s.thread = _FakeThread()
    s.stop_flag = False
    s.max_mhz = 2070.0
    s.samples = samples
    s.window = window
    return s


def test_clock_record_keeps_only_the_timed_window_and_decodes_reasons():
    samples = [
        (0.5, 900.0, 0x1),          # before the window (idle): dropped
        (1.0, 2070.0, 0x0),
        (1.1, 1800.0, 0x4),         # sw_power_cap
        (1.2, 1500.0, 0x4 | 0x8),   # + hw_slowdown
        (2.5, 300.0, 0x40),         # after the window: dropped
    ]
    s = _sampler(samples, (1.0, 1.2))
    rec = s.stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 1800.0
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s.stop_flag and s.lib.shutdown == 1


def test_clock_record_is_none_without_samples_in_the_window():
    s = _sampler([(0.1, 2070.0, 0), (9.0, 2070.0, 0)], (1.0, 2.0))
    assert s.stop() is None


def test_thermal_reasons_are_named():
    s = _sampler([(1.0, 1200.0, 0x20 | 0x40)], (0.0, 2.0))
    assert s.stop()["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_sampler_falls_back_to_nvidia_smi(monkeypatch):
    class _NoNvml:
        def __init__(self, index):
            raise OSError("no libnvidia-ml")
    monkeypatch.setattr(bench, "NvmlClockSampler", _NoNvml)
    s = bench.clock_sampler(0)
    assert isinstance(s, bench.ClockSampler)
    s.mark(0.0, 1.0)   # accepted and ignored: nvidia-smi samples are not timestamped here


def test_algorithmic_bytes_per_format():
    # 4-bit: half a byte a weight + one absmax code a block + one fp32 a group
    assert bench.packed_bytes(4096, 4096) == 4096 * 4096 // 2 + 4096 * 64 + 4 * 1024
    # int8: a byte a weight + one fp32 absmax a block
    assert bench.packed_bytes(4096, 4096, "int8") == 4096 * 4096 + 4 * 4096 * 64
    from dequant_gemm_gb300 import workloads as wl
    p = wl.WORKLOADS["prefill_up_11008x4096_bf16"].projections[0]
    w = wl.WORKLOADS["prefill_up_11008x4096_bf16"]
    f, b = bench.fwd_work(p, 4096, w)
    assert f == 2 * 4096 * 11008 * 4096
    assert b == bench.packed_bytes(11008, 4096) + 2 * 4096 * 4096 + 2 * 4096 * 11008
    assert bench.quant_bytes(p, w) == 2 * 11008 * 4096 + bench.packed_bytes(11008, 4096)


def test_class_record_roofline():
    pk = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    # 1 TFLOP and 1 GB in 1 ms: 1000 TFLOP/s (0.5 of burst), 1000 GB/s
    r = bench.class_record(1e12, 1e9, 1e-3, pk)
    assert r["bound"] == "tensor" and abs(r["tensor_frac_burst"] - 0.5) < 1e-12
    assert abs(r["tensor_frac_sustained"] - 0.625) < 1e-12
    assert abs(r["roofline_frac"] - 0.5) < 1e-12
    # memory-bound: 8 GB in 2 ms at 8000 GB/s peak is half the copy bandwidth
    r = bench.class_record(1e9, 8e9, 2e-3, pk)
    assert r["bound"] == "hbm" and abs(r["hbm_frac"] - 0.5) < 1e-12 and abs(r["roofline_frac"] - 0.5) < 1e-12


def _call_list(name, group=True, parallel_tc=True):
    """The call list of a workload's step without device buffers."""
    from dequant_gemm_gb300 import workloads as wl
    st = object.__new__(bench.Step)
    st.nf4 = None
    st.w = wl.WORKLOADS[name]
    st.rotate = 1
    st.group_small_m = group
    st.parallel_tc = parallel_tc
    st.x, st.y, st.dy, st.dx, st.q, st.wcopies = {}, {}, {}, {}, [[None] * 7], [[None] * 7]
    st.calls = st._calls()
    return st


def test_layer_step_groups_small_m_forwards_and_counts_x_once():
    st = _call_list("qwen2.5_7b_layer")
    P = st.w.projections
    m1 = [c for c in st.calls if c[0] == "fwd_M1"]
    assert [c[6] for c in m1] == [(0, 1, 2), 3, (4, 5), 6]
    for c in m1:
        js = c[6] if isinstance(c[6], tuple) else (c[6],)
        f = sum(bench.fwd_work(P[j], 1, st.w)[0] for j in js)
        b = sum(bench.fwd_work(P[j], 1, st.w)[1] for j in js) - (len(js) - 1) * 2 * P[js[0]].cols
        assert (c[1], c[2]) == (f, b)
    # the same work either way
    sep = _call_list("qwen2.5_7b_layer", group=False)
    assert sum(c[1] for c in st.calls) == sum(c[1] for c in sep.calls)
    assert len([c for c in sep.calls if c[0] == "fwd_M1"]) == 7
    # tensor-core calls of an input group share a stream group tag only when parallel
    tags = {c[5] for c in st.calls if c[0] == "fwd_M2048"}
    serial = {c[5] for c in _call_list("qwen2.5_7b_layer", parallel_tc=False).calls
              if c[0] == "fwd_M2048"}
    assert len(tags) == 4 and len(serial) == 7


def test_end_to_end_schedule_copies_every_output_once_after_its_writer():
    st = _call_list("qwen2.5_7b_layer")
    P = st.w.projections
    order = sorted(range(len(P)), key=lambda i: -P[i].rows * P[i].cols)
    turn, out_turn = st.e2e_schedule(order)
    pos = {i: n for n, i in enumerate(order)}
    expected = {(k, j, M) for j in range(len(P)) for k, ms in (("fwd", st.w.fwd_m), ("dx", st.w.dx_m))
                for M in ms}
    assert set(out_turn) == expected
    for c, t in zip(st.calls, turn):
        js = c[6] if isinstance(c[6], tuple) else (c[6],)
        assert t == max(pos[j] for j in js)          # after every weight it reads has landed
        for kind in ("fwd", "dx"):
            if c[0].startswith(kind + "_M"):
                for j in js:
                    assert out_turn[(kind, j, int(c[0][len(kind) + 2:]))] >= t
