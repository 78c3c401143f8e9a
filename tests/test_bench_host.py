"""Host-side pieces of bench.py that its JSON line rests on: the algorithmic
work and bytes behind the roofline figures (counted here from the products'
shapes and the tensors' sizes), the clock sampler's parsing of nvidia-smi
output, and the source hash that retires a recorded ncu traffic figure once a
kernel's code changes.  No GPU needed."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_chunked_flops_from_product_shapes(bench):
    """Per chunk of C tokens: per key head the two Gram products, per value head
    the WY products and the state-pass products; the triangular solve apart."""
    C, h_k, h_v, d_k, d_v = 64, 16, 32, 128, 128
    mma = lambda m, n, k: 2 * m * n * k
    per_key = mma(C, C, d_k) + mma(C, C, d_k)                      # K K^T, Q K^T
    per_val = (mma(C, d_k, C) + mma(C, d_v, C)                    # W, U~
               + mma(C, d_v, C)                                    # P U
               + mma(C, d_v, d_k) + mma(C, d_v, d_k)               # W S^T, Q S^T
               + mma(d_v, d_k, C))                                 # state update
    want = (h_k * per_key + h_v * per_val) / C
    got = bench.chunked_flops_per_token(h_k, h_v, d_k, d_v)
    assert got == pytest.approx(want, rel=1e-12)
    assert round(got) == 5_242_880                                  # the figure the roofline uses
    assert got * 4096 == pytest.approx(21.47e9, rel=1e-3)
    solve = bench.solve_flops_per_token(h_v)                        # C^3 / 3 MACs per chunk
    assert solve == pytest.approx(h_v * (2 * C ** 3 // 3) / C, rel=1e-12)
    assert round(got + solve) == 5_330_261


def test_bytes_from_tensor_sizes(bench):
    T, N, h_k, h_v, d = 4096, 1, 16, 32, 128
    q = k = T * h_k * d * 2
    v = o = T * h_v * d * 2
    g = beta = T * h_v * 4
    state_out = N * h_v * d * d * 4
    assert bench.prefill_bytes(T, N, h_k, h_v, d, d, 2, False) == q + k + v + o + g + beta + state_out
    assert bench.prefill_bytes(T, N, h_k, h_v, d, d, 2, True) == (q + k + v + o + g + beta
                                                                 + 2 * state_out)
    B = 256
    decode = 2 * B * h_v * d * d * 4 + 2 * B * h_k * d * 2 + 2 * B * h_v * d * 2 + 2 * B * h_v * 4
    assert bench.decode_bytes(B, h_k, h_v, d, d, 2) == decode == 1_080_098_816
    assert bench.scan_flops_per_token(h_v, d, d) == 6 * d * d * h_v


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_parses_smi_lines(bench, tmp_path):
    path = tmp_path / "clocks.csv"
    lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1010.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    path.write_text("\n".join(lines) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path, s.out = _FakeProc(), str(path), open(os.devnull, "w")
    r = s.stop()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    assert not path.exists()


def test_clock_sampler_reports_throttle_reasons(bench, tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("0, 1500, 2070, 1400.0, 0x8, Active, Not Active, Active, Not Active\n")
    s = bench.ClockSampler(0)
    s.proc, s.path, s.out = _FakeProc(), str(path), open(os.devnull, "w")
    r = s.stop()
    assert r["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and r["sm_mhz"] == 1500.0


def test_source_hash_ignores_comments_but_not_code(bench, tmp_path, monkeypatch):
    csrc = tmp_path / "gated_deltanet_linear_recurrence_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    f.write_text("int a = 1;  // one\n/* block\n comment */\nint b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash(["k.cu"])
    f.write_text("// header\nint a = 1;  // changed comment\n\nint b = 2;\n")
    assert bench.source_hash(["k.cu"]) == h0
    f.write_text("int a = 1;\nint b = 3;\n")
    assert bench.source_hash(["k.cu"]) != h0


def test_recorded_traffic_matches_the_current_sources(bench):
    """Every ncu figure the bench can report has its summary under profiles/,
    and a record whose kernel sources changed since its capture is reported as
    null, never as a number."""
    for name, rec in bench.NCU_TRAFFIC.items():
        assert os.path.exists(os.path.join(ROOT, rec["profile"])), rec["profile"]
        fresh = bench.source_hash(rec["files"]) == rec["sha256_16"]
        assert bench.ncu_traffic(name) == (rec["bytes"] if fresh else None)


def test_sweep_thresholds(bench):
    """The crossover table's thresholds: the smallest swept length from which
    the faster form of each pair stays faster at every longer length."""
    rows = {
        8: {"scan": 5.0, "chunked_fused": 9.0, "chunked_split": 12.0, "chunked_coop": 20.0},
        16: {"scan": 9.0, "chunked_fused": 8.0, "chunked_split": 11.0, "chunked_coop": 19.0},
        32: {"scan": 12.0, "chunked_fused": 9.0, "chunked_split": 8.0, "chunked_coop": 9.0},
        64: {"scan": 20.0, "chunked_fused": 12.0, "chunked_split": 13.0, "chunked_coop": 11.0},
        128: {"chunked_fused": 20.0, "chunked_split": 15.0, "chunked_coop": 14.0},
    }
    forms = ["scan", "chunked_fused", "chunked_split", "chunked_coop"]
    th = bench.sweep_thresholds(rows, forms)
    # scan loses from 16; split beats fused at 32, loses at 64, wins again from 128;
    # coop beats split from 64
    assert th == {"scan_below": 16, "split_from_avg": 128, "coop_from_avg": 64}
    # no fused kernel (d_k = 64): no fused threshold; no cooperative form: None
    th2 = bench.sweep_thresholds({L: {k: v for k, v in r.items() if k not in
                                      ("chunked_fused", "chunked_coop")}
                                  for L, r in rows.items()}, ["scan", "chunked_split"])
    assert th2 == {"scan_below": 32, "split_from_avg": 0, "coop_from_avg": None}
