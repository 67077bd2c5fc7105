"""The benchmark's bookkeeping, on the CPU: workload shapes and chaining, the
algorithmic bytes its GB/s divide by, and its oracle timing helper."""
import bench
from weight_streaming_skinny_gb300 import inputs


def _fp8_weight_bytes(N, K):
    return N * K + 4 * ((N + 127) // 128) * ((K + 127) // 128)


def test_model_workload_shapes_and_bytes():
    specs, cfg = bench.layer_specs("qwen72b_model_fp8_m1")
    assert cfg == 4 and len(specs) == 4 * 80 + 1
    assert [s[5].split(".")[0] for s in specs[:4]] == ["qkv", "o", "gate_up", "down"]
    assert [s[6] for s in specs[:4]] == [0, 0, 1, 0]              # SwiGLU on gate_up
    assert specs[-1][:4] == ("bf16", 1, 152064, 8192) and specs[-1][6] == 2
    # algorithmic bytes per token written out from the shapes: weights (+ block
    # scales) + x + y (+ bias); SwiGLU writes N/2 columns, the argmax M ids
    layer = (_fp8_weight_bytes(10240, 8192) + 2 * 8192 + 2 * 10240 + 2 * 10240
             + _fp8_weight_bytes(8192, 8192) + 2 * 8192 + 2 * 8192
             + _fp8_weight_bytes(59136, 8192) + 2 * 8192 + 2 * 59136 // 2
             + _fp8_weight_bytes(8192, 29568) + 2 * 29568 + 2 * 8192)
    lm_head = 2 * 152064 * 8192 + 2 * 8192 + 4
    total = 0
    for dt, M, N, K, bias, name, act in specs:
        L = inputs.LayerInputs(dt, M, N, K, None, None, None, object() if bias else None)
        L.act = act
        total += bench.out_bytes(L)
    assert total == 80 * layer + lm_head == 72740515844


def test_decoder_workload_is_the_model_first_layer():
    model, _ = bench.layer_specs("qwen72b_model_fp8_m1")
    dec, cfg = bench.layer_specs("qwen72b_decoder_fp8_m1")
    assert cfg == 4 and dec == model[:4]
    lm, _ = bench.layer_specs("qwen72b_lm_head_bf16_m1")
    assert lm == [model[-1]]


def test_layer_and_sweep_workloads():
    for wl, dt, M in (("qwen72b_layer_bf16_m1", "bf16", 1), ("qwen72b_layer_fp8_m6", "fp8_b128", 6)):
        specs, _ = bench.layer_specs(wl)
        assert [(s[0], s[1], s[2], s[3], s[4]) for s in specs] == [
            (dt, M, 10240, 8192, True), (dt, M, 8192, 8192, False),
            (dt, M, 59136, 8192, False), (dt, M, 8192, 29568, False)]
    for m in bench.MLP_TOKENS:
        specs, cfg = bench.layer_specs(f"qwen72b_mlp_fp8_m{m}")
        assert cfg == 3 and [(s[1], s[2], s[3]) for s in specs] == [(m, 59136, 8192), (m, 8192, 29568)]


def test_model_chaining_on_cpu_shapes():
    """The model chains down -> next qkv, o -> gate_up, gate_up -> down and the
    last down -> lm_head; o keeps its own x (the attention output stand-in)."""
    specs, _ = bench.layer_specs("qwen72b_model_fp8_m1")
    chained = []
    for i in range(1, len(specs)):
        prev, cur = specs[i - 1], specs[i]
        out_cols = prev[2] // 2 if prev[6] == 1 else prev[2]
        if out_cols == cur[3] and prev[1] == cur[1] and cur[5].split(".")[0] != "o":
            chained.append(cur[5].split(".")[0])
    assert len(chained) == 3 * 80
    assert chained.count("gate_up") == 80 and chained.count("down") == 80
    assert chained.count("qkv") == 79 and chained.count("lm_head") == 1


def test_dtype_labels():
    for wl in bench.WORKLOADS:
        specs, _ = bench.layer_specs(wl)
        label = bench.dtype_label(wl, specs)
        if {s[0] for s in specs} == {"bf16"}:
            assert label == "bf16"
        else:
            assert "fp8_e4m3" in label and "fp32 accumulate" in label


def test_cpu_oracle_timing_helper_on_a_tiny_sample():
    layers = []
    for i, (dt, act) in enumerate(((inputs.DTYPE_BF16, 0), (inputs.DTYPE_FP8_B128, 1),
                                   (inputs.DTYPE_BF16, 2))):
        L = inputs.make_layer(dt, 1, 256, 256, bias=(i == 0), config_id=0, layer_idx=i)
        L.act = act
        layers.append((f"l{i}", L))
    gbs, threads, passes, t = bench.cpu_oracle_gbs(layers, 0.0, 0.5, threads=1)
    assert threads == 1 and passes == 1 and gbs > 0 and t > 0


def test_percentiles():
    vals = [float(v) for v in range(11)]
    assert bench._pctl(vals, 0.1) == 1.0 and bench._pctl(vals, 0.9) == 9.0
    d = bench._dist_us([0.001, 0.002, 0.003])
    assert d["median_us"] == 2.0 and d["n"] == 3


def test_cold_copies_cover_three_l2():
    l2 = 129 * 10**6
    for dt, N, K, bias, want in (("bf16", 10240, 8192, True, 3), ("fp8_b128", 8192, 8192, False, 6),
                                 ("bf16", 59136, 8192, False, 1), ("bf16", 1024, 1024, True, 184)):
        L = inputs.LayerInputs(dt, 1, N, K, None, None, None, object() if bias else None)
        n = bench.cold_copies(L, l2)
        assert n == want and n * L.algorithmic_bytes >= 3 * l2
        assert n == 1 or (n - 1) * L.algorithmic_bytes < 3 * l2
