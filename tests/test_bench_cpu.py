"""Host-side pieces of bench.py without a GPU: the FLOP convention, the
traffic lookup that goes stale when a kernel source changes, the reference
arm (the fp64 oracle on the host cores) and its JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_flop_convention_by_hand():
    """4 N L d per head forward (L = key bound), halved under causal, times the
    nonzero-block fraction under a block mask; backward 2.5x, step 3.5x."""
    s = W.SPECS["gpt2"]                      # B8 H12 N1024 d64 causal
    fl = bench.counted_flops(s, None)
    want = 4.0 * 1024 * 1024 * 64 * 12 * 8 / 2
    assert fl["fwd"] == want and fl["bwd"] == 2.5 * want and fl["step"] == 3.5 * want
    kv = np.array([256, 300, 512, 1000], np.int32)   # clamped to N = 512
    b = W.Spec("t", 4, 2, 512, 64, False, 0.125)
    fl = bench.counted_flops(b, kv)
    assert fl["fwd"] == sum(4.0 * 512 * min(L, 512) * 64 * 2 for L in kv)
    assert fl["nominal_step"] == 3.5 * 4.0 * 512 * 512 * 64 * 2 * 4
    mask = np.zeros((4, 4), np.uint8)
    mask[0, 0] = mask[1, 2] = mask[3, 3] = 1
    c = W.Spec("m", 1, 1, 512, 64, False, 0.125)
    assert bench.counted_flops(c, None, mask)["fwd"] == 4.0 * 512 * 512 * 64 * 3 / 16
    d128 = W.Spec("w", 1, 1, 256, 128, False, 0.125)
    assert bench.counted_flops(d128, None)["fwd"] == 4.0 * 256 * 256 * 128


def test_traffic_lookup_goes_stale_with_the_sources(monkeypatch):
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    entries = json.load(open(path))
    key = "fa_bwd_main_kernel:bert"
    assert bench.load_traffic("fa_bwd_main_kernel", "bert") in (None, entries[key]["bytes"])
    monkeypatch.setattr(bench, "_sources_hash", lambda names: entries[key]["sources"])
    assert bench.load_traffic("fa_bwd_main_kernel", "bert") == entries[key]["bytes"]
    monkeypatch.setattr(bench, "_sources_hash", lambda names: "0" * 16)
    assert bench.load_traffic("fa_bwd_main_kernel", "bert") is None
    assert bench.load_traffic("no_such_kernel", "bert") is None


def test_every_captured_kernel_names_existing_sources():
    csrc = os.path.join(ROOT, "exact_io_aware_25_gb300", "csrc")
    for kernel, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), (kernel, n)


def test_workload_config_names_the_workload():
    for name in ("tiny", "bert", "gpt2", "gpt2_4k"):
        w = W.make(name, B=1, H=1, N=256) if name != "tiny" else W.make(name)
        cfg = bench.workload_config(w)
        assert cfg["workload"] and cfg["d"] == 64 and "flushed" in cfg["l2"]
    cfg = bench.workload_config(W.make("tiny"), dropout=0.25, seed=7)
    assert cfg["dropout"]["p"] == 0.25 and cfg["dropout"]["seed"] == 7


def test_reference_arm_prints_one_json_line(fa_lib, oracle_mod):
    """`bench.py --impl reference` runs the oracle on the host cores and
    prints the contract's line with impl, cpu_baseline and e2e."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["higher_is_better"] is True and d["steps"] == 1


def test_traffic_hash_ignores_comments_but_not_code():
    """The staleness check hashes what the compiler sees: comments and
    whitespace may change, code and string literals may not."""
    a = 'int x = 1; // note\n/* block */ asm("add.f32 %0, %1; // not a comment");\n'
    b = 'int x = 1;   /* reworded note */\n\n asm("add.f32 %0, %1; // not a comment");'
    c = 'int x = 2; asm("add.f32 %0, %1; // not a comment");'
    d = 'int x = 1; asm("add.f32 %0, %1; // changed");'
    assert bench._code_text(a) == bench._code_text(b)
    assert bench._code_text(a) != bench._code_text(c)
    assert bench._code_text(a) != bench._code_text(d)
    assert bench._code_text("char q = '\\''; // x") == "char q = '\\'';"


def test_allowed_keys_is_the_support_of_the_oracles_probabilities(oracle_mod):
    """The reference arm's row sample counts 10*L*d per row with L from
    bench.allowed_keys: L must be the number of keys with nonzero P in the
    oracle, for every mask kind (ragged N, causal, key padding, block mask)."""
    rng = np.random.default_rng(5)
    mask = (rng.random((3, 3)) < 0.5).astype(np.uint8)
    mask[2, 0] = 1
    for causal, kv, bm in [(False, None, None), (True, None, None),
                           (False, np.array([300, 137], np.int32), None),
                           (True, np.array([251, 300], np.int32), mask),
                           (False, None, mask)]:
        w = W.make("tiny", seed=8, B=2, H=1, N=300, causal=causal)
        q, k = w.f64("q"), w.f64("k")
        for b in range(2):
            P = oracle_mod.probs(q, k, w.spec.scale, bh=b, causal=causal, kv_len=kv,
                                 block_mask=bm)
            for i in range(300):
                want = int(np.count_nonzero(P[i]))
                assert bench.allowed_keys(w.spec, kv, bm, b, i) == want, (causal, b, i)


def test_reference_row_sample_counts_its_rows(oracle_mod):
    w = W.make("tiny", seed=9, B=1, H=2, N=256, causal=True)
    rows = np.array([0, 5, 255, 256 + 17], np.int64)
    f, t, threads = bench.time_oracle_rows(w, rows)
    assert t > 0 and threads >= 1
    assert f == 10.0 * 64 * sum([1, 6, 256, 18])


def test_oracle_head_timer_runs_the_heads_it_is_asked_for(oracle_mod):
    """time_oracle with max_units bounds the heads, and an unlimited budget
    does not stop it before the first one (the reference arm sizes its steps
    from one timed head)."""
    w = W.make("tiny", B=1, H=3, N=64)
    f, t, heads, _ = bench.time_oracle(w, float("inf"), max_units=1)
    assert heads == 1 and t > 0 and f > 0
    f2, _, heads2, _ = bench.time_oracle(w, float("inf"), max_units=2)
    assert heads2 == 2 and f2 == pytest.approx(2 * f)
    assert bench.time_oracle(w, 0.0)[2] == 0
