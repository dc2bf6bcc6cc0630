"""Host-side logic that needs no GPU: the load-time weight layout of model.py,
and the measurement helpers of bench.py (clock sampling, peaks, the ncu
traffic lookup)."""
import hashlib
import json

import numpy as np
import pytest
import torch

import oracle as O
import seeded_inputs as si


def _checkpoint(m, layer=0):
    names = si.weight_names(layer) + [f"layer{layer}.{x}" for x in
                                      ("input_layernorm", "post_attention_layernorm", "q_norm", "k_norm")]
    return {n: si.checkpoint_tensor(m, n, seed=3) for n in names}


@pytest.mark.parametrize("tp", [1, 2, 4])
def test_shard_layer_matches_the_oracle_layout(tp):
    """model.shard_layer stacks the shards exactly as the oracle's
    QKVParallelLinear / MergedColumnParallelLinear rank weights, and its
    row-split o_proj / down_proj reproduce the oracle's shard-summed Linear."""
    from qwen3_transformer_forward_gb300 import model as M
    m = si.TINY.replace(n_heads=8, n_kv_heads=4, tp=tp)
    ck = _checkpoint(m)
    lp = M.shard_layer(m, ck, 0, "cpu")
    np_ = {k: v.double().numpy() for k, v in ck.items()}
    qkv_ref = np.concatenate([O.qkv_shard_weight(np_["layer0.q_proj"], np_["layer0.k_proj"], np_["layer0.v_proj"],
                                                 m.n_heads, m.n_kv_heads, m.head_dim, tp, r) for r in range(tp)])
    assert np.array_equal(lp.qkv.double().numpy(), qkv_ref)
    gu_ref = np.concatenate([O.gate_up_shard_weight(np_["layer0.gate_proj"], np_["layer0.up_proj"], tp, r)
                             for r in range(tp)])
    assert np.array_equal(lp.gate_up.double().numpy(), gu_ref)
    x = si.normal(5, "host.x", (3, m.q_size), 1.0, "f32").double().numpy()
    xi = si.normal(5, "host.xi", (3, m.intermediate), 1.0, "f32").double().numpy()
    for w_st, w_full, xx in ((lp.o, np_["layer0.o_proj"], x), (lp.down, np_["layer0.down_proj"], xi)):
        k_l = xx.shape[1] // tp
        assert tuple(w_st.shape) == (tp, w_full.shape[0], k_l)
        shards = [xx[:, r * k_l:(r + 1) * k_l] for r in range(tp)]
        got = sum(shards[r] @ w_st[r].double().numpy().T for r in range(tp))
        np.testing.assert_allclose(got, O.row_parallel_linear(shards, w_full, tp, "f64"), rtol=1e-12, atol=1e-12)
    for n, attr in (("input_layernorm", "input_ln"), ("post_attention_layernorm", "post_ln"), ("q_norm", "q_norm"),
                    ("k_norm", "k_norm")):
        assert torch.equal(getattr(lp, attr), ck[f"layer0.{n}"])


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _sampler_with(tmp_path, lines):
    import bench
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("".join(line + "\n" for line in lines))
    s.proc = _FakeProc()
    return s


def test_clock_sampler_median_and_reasons(tmp_path):
    na = "Not Active"
    rows = [f"0, 2070, 2070, 810.5, 0x0000000000000000, {na}, {na}, {na}, {na}",
            f"0, 1965, 2070, 1391.0, 0x0000000000000004, {na}, {na}, {na}, Active",
            f"0, 2070, 2070, 902.0, 0x0000000000000000, {na}, {na}, {na}, {na}",
            "0, [N/A]"]   # a short line is skipped
    c = _sampler_with(tmp_path, rows).stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3


def test_clock_sampler_flags_thermal_slowdown_and_empty_runs(tmp_path):
    na = "Not Active"
    c = _sampler_with(tmp_path, [f"0, 1500, 2070, 1300, 0x40, {na}, Active, {na}, {na}"]).stop()
    assert c["reasons"] == ["hw_thermal_slowdown"] and c["sm_mhz"] == 1500.0
    assert _sampler_with(tmp_path, []).stop()["reasons"] == ["no samples"]
    import bench
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]


def test_load_peaks_measured_and_fallback(tmp_path, monkeypatch):
    import bench
    mp = {"hbm_gbs": 6000.5, "bf16_tflops": 1900.25, "bf16_tflops_sustained": 1700.75}
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(mp))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm"] == 6000.5
    assert p["tensor"] == 1700.75 and p["tensor_burst"] == 1900.25   # sustained for kernels inside the step
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.load_peaks()["source"] == "fallback"


def test_profile_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    import bench
    src = tmp_path / "qwen3_transformer_forward_gb300" / "csrc"
    src.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    code = b"// kernel source as captured\n"
    (src / "attention.cu").write_bytes(code)
    (tmp_path / "profiles" / "k.json").write_text(json.dumps(
        {"dram_bytes_per_launch": 69676000,
         "sources_sha1": {"qwen3_transformer_forward_gb300/csrc/attention.cu": hashlib.sha1(code).hexdigest()}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k") == 69676000
    assert bench.profile_traffic("missing") is None
    (src / "attention.cu").write_bytes(code + b"// changed since\n")
    assert bench.profile_traffic("k") is None


def test_max_over_ranks_is_identity_on_one_rank():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
