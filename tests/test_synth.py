"""The seeded input recipe on CPU (not gpu): the distributions, shapes and
seeding that the synthetic workloads are stated to have."""
import numpy as np
import pytest

from bit_quantized_linear_gb300 import synth


def test_seeding_is_deterministic_and_keyed():
    a = synth.rng_for("w", 0, "t", "weight").standard_normal(8)
    b = synth.rng_for("w", 0, "t", "weight").standard_normal(8)
    assert np.array_equal(a, b)
    for other in [("w", 1, "t", "weight"), ("w", 0, "u", "weight"), ("w", 0, "t", "act"), ("v", 0, "t", "weight")]:
        assert not np.array_equal(a, synth.rng_for(*other).standard_normal(8)), other


def test_bf16_rounding_is_nearest_even():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)  # BF16 spacing in [1, 2)
    x = np.array([one, one + ulp / 2, one + 3 * ulp / 2, one + ulp / 4, -(one + 3 * ulp / 2), 3.0e38],
                 np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))
    want = np.array([1.0, 1.0, 1.0 + 2 * ulp, 1.0, -(1.0 + 2 * ulp)], np.float32)
    assert np.array_equal(got[:5], want)                 # ties go to the even neighbour
    assert np.isfinite(got[5]) and abs(float(got[5]) / 3.0e38 - 1) <= 2 ** -9  # large values: half-ulp rounding


def test_weight_recipe():
    N, K = 512, 2048
    w = synth.weights(N, K, synth.rng_for("t", 0, "w", "weight"))
    assert w.dtype == np.float32 and w.shape == (N, K)
    assert abs(float(w.mean())) < 5e-4
    assert float(w.std()) == pytest.approx(1.0 / np.sqrt(K), rel=0.01)


def test_activation_recipe_with_outlier_channels():
    M, K = 2048, 1000
    rng = synth.rng_for("t", 0, "x", "act")
    outl = synth.outlier_channels(K, synth.rng_for("t", 0, "x", "outliers"))
    assert outl.size == 10 and np.all(np.diff(outl) > 0) and outl.max() < K   # round(K / 100), distinct
    x = synth.bf16_bits_to_f32(synth.activations(M, K, rng, outl))
    plain = np.setdiff1d(np.arange(K), outl)
    assert float(x[:, plain].std()) == pytest.approx(1.0, rel=0.02)
    assert float(x[:, outl].std()) == pytest.approx(20.0, rel=0.05)
    # BF16 values: the low 16 bits of every fp32 pattern are zero
    assert not np.any(x.view(np.uint32) & np.uint32(0xFFFF))


def test_activations_are_the_same_in_row_chunks():
    K = 64
    a = synth.activations(10, K, synth.rng_for("t", 0, "x", "act"), chunk_rows=3)
    b = synth.activations(10, K, synth.rng_for("t", 0, "x", "act"), chunk_rows=4096)
    assert np.array_equal(a, b)


def test_bias_recipe():
    b = synth.bf16_bits_to_f32(synth.bias(20000, synth.rng_for("t", 0, "b", "bias")))
    assert float(b.std()) == pytest.approx(0.1, rel=0.03)


def test_workload_shapes():
    d = synth.workload(synth.DECODE7B).linears
    assert len(d) == 15 and sorted({l.M for l in d}) == [1, 8, 32, 128, 256]
    assert {(l.name, l.K, l.N) for l in d} == {("q_proj", 3584, 3584), ("gate_up_proj", 3584, 37888),
                                                ("down_proj", 18944, 3584)}
    assert all(l.qtype == "e4m3" and l.form == "w8a16" and l.outliers for l in d)
    p = synth.workload(synth.PREFILL).linears
    assert len(p) == 12 and sorted({l.M for l in p}) == [1024, 4096, 16384, 32640]
    assert all(l.qtype == "e4m3" and l.form == "w8a8" for l in p)
    w = synth.workload(synth.W8A8_3B).linears
    assert all(l.qtype == "int8" and l.form == "w8a8" and l.bias for l in w)
    s = synth.workload(synth.SMALL).linears
    assert [(l.M, l.K, l.N) for l in s] == [(1, 1024, 1024), (16, 1024, 1024)]
    sd, sp = synth.stack_linears("decode"), synth.stack_linears("prefill")
    assert len(sd) == len(sp) == 36 * 6
    assert {l.M for l in sd} == {256} and {l.M for l in sp} == {8192}
    sf = synth.stack_linears("decode", fused=True)
    assert len(sf) == 36 * 4 and sum(l.glu for l in sf) == 36
    glu = [l for l in sf if l.glu][0]
    assert (glu.K, glu.N) == (2048, 2 * 11008)


def test_kv_slots():
    for layer in (0, 27):
        ctx = synth.kv_context_slots(layer)
        chunk = synth.kv_chunk_slots(layer)
        assert ctx.size == synth.KV_CONTEXT and np.unique(ctx).size == ctx.size
        assert ctx.min() == 0 and ctx.max() == synth.KV_CONTEXT - 1
        assert chunk.size == synth.KV_CHUNK and np.array_equal(chunk, ctx[:synth.KV_CHUNK])
        # tokens are contiguous inside each 256-token block
        blocks = chunk.reshape(-1, synth.KV_BLOCK)
        assert np.all(np.diff(blocks, axis=1) == 1) and np.all(blocks[:, 0] % synth.KV_BLOCK == 0)
    assert not np.array_equal(synth.kv_block_table(0), synth.kv_block_table(1))
    k = synth.kv_tokens(0, 64, "k")
    assert k.shape == (64, synth.KV_HEADS * synth.KV_HEAD_DIM) and k.dtype == np.uint16
