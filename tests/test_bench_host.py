"""Host-side logic of bench.py (no GPU): the whole-step roofline's algorithmic
work on a hand-checked packed row, the code hash that ties an ncu capture to
the GEMM sources, and the committed capture's per-launch traffic lookup."""
import dataclasses

import numpy as np

import bench


@dataclasses.dataclass
class _Cfg:
    d: int = 64
    ffn: int = 96
    V: int = 100
    D: int = 1


def test_step_roofline_counts_state_rows_and_visible_pairs():
    # one packed row: segments 0 (t = 0..2), 1 (t = 3, 4), pad (t = 5).  Depth 1 has state at
    # t = 0, 1 (next token in the same segment) and t = 3; t = 2 and t = 4 end their segments.
    seg = np.array([[0, 0, 0, 1, 1, -1]], dtype=np.int32)
    cfg = _Cfg()
    peaks = {"bf16_tflops": 1.0, "hbm_gbs": 1.0}  # 1e12 FLOP/s, 1e9 B/s
    r = bench.step_roofline(cfg, seg, [5.0, 2.0], 1000.0, 1.0, peaks)
    rows, pairs = 3, 1 + 2 + 1  # keys from the segment start to t: 1, 2 and 1
    d, f, V = cfg.d, cfg.ffn, cfg.V
    t = r["terms_ms"]
    assert np.isclose(t["gemm_block"], rows * (12 * d * d + 6 * d * f) / 1e12 * 1e3)
    # attention: the larger of its FLOPs (4 d per visible pair) and its bytes (q, k, v read and
    # o written in bf16 per row with state)
    assert np.isclose(t["attention"], max(4 * d * pairs / 1e12, rows * 8 * d / 1e9) * 1e3)
    assert np.isclose(t["head_ce"], 2 * d * V * 7.0 / 1e12 * 1e3)
    assert np.isclose(t["norms_prologue"], rows * (8 * d + 8 * d) / 1e9 * 1e3)
    assert np.isclose(t["head_norms"], 4 * d * 7.0 / 1e9 * 1e3)
    assert np.isclose(t["spec_verify"], 1000.0 / 1e9 * 1e3)
    assert np.isclose(r["roofline_ms"], sum(t.values()))
    assert np.isclose(r["frac"], r["roofline_ms"] / 1.0)


def test_step_roofline_depth_two_drops_segment_tails():
    # depth 2 needs t + 2 in t's segment: in a 4-token segment that is t = 0, 1 only
    seg = np.array([[7, 7, 7, 7]], dtype=np.int32)
    cfg = _Cfg(D=2)
    peaks = {"bf16_tflops": 1.0, "hbm_gbs": 1.0}
    r = bench.step_roofline(cfg, seg, [0.0, 0.0, 0.0], 0.0, 1.0, peaks)
    rows = 3 + 2  # depth 1: t = 0, 1, 2; depth 2: t = 0, 1
    pairs = (1 + 2 + 3) + (1 + 2)
    assert np.isclose(r["terms_ms"]["gemm_block"], rows * (12 * cfg.d ** 2 + 6 * cfg.d * cfg.ffn) / 1e9)
    assert np.isclose(r["terms_ms"]["attention"], max(4 * cfg.d * pairs / 1e9, rows * 8 * cfg.d / 1e6))


def test_code_lines_ignores_comments_and_blank_lines():
    a = "int x = 1;  // one\n\n  // a whole comment line\nint y = 2;\n"
    b = "int x = 1;\nint y = 2;   // two\n"
    assert bench.code_lines(a) == bench.code_lines(b) == "int x = 1;\nint y = 2;"
    # a // inside a string literal is code
    assert bench.code_lines('asm("a // b"); // c') == 'asm("a // b");'
    assert bench.code_lines("x = 1;") != bench.code_lines("x = 2;")


def test_capture_lookup_is_keyed_by_the_gemm_code():
    # the head-GEMM ncu summary is keyed by the hash of the GEMM code it was taken on; the
    # lookup returns its per-launch DRAM bytes exactly when that key is the current code's
    import re
    text = open(bench.HEAD_PROFILE, encoding="utf-8").read()
    key = re.search(r"^- kernel_source_sha256: `([0-9a-f]{16})`$", text, re.M).group(1)
    dram = float(re.search(r"^- dram_bytes_per_launch: `(\d+)`$", text, re.M).group(1))
    if key == bench.gemm_source_hash():
        assert bench.recorded_traffic() == dram
    else:
        assert bench.recorded_traffic() is None
