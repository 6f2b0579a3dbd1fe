"""Host logic of bench.py's measurement accounting: the algorithmic cache
bytes every GB/s figure and the roofline's `achieved` divide by, the
context each step decodes over, and the rule that the recorded ncu traffic
is reported only while the decode sources still hash to the recorded value.
No GPU involved."""
import bench


def test_row_bytes_per_cell_and_kv_head():
    # K and V codes, plus an fp16 scale per 64 dims (int8) or, for K8V4,
    # int8 K + its per-64 scales and 4-bit V + an fp16 scale per 32 dims
    assert bench._row_bytes("f16", 128) == 2 * 128 * 2
    assert bench._row_bytes("q8", 128) == 2 * (128 + 2 * 2)
    assert bench._row_bytes(True, 128) == bench._row_bytes("q8", 128)
    assert bench._row_bytes(False, 128) == bench._row_bytes("f16", 128)
    assert bench._row_bytes("k8v4", 128) == 128 + 2 * 2 + 64 + 2 * 4 == 204
    assert bench._row_bytes("k8v4", 256) == 408
    # the gqa32k decode at 32768 cells, 8 KV heads: the per-call bytes the
    # design notes quote
    assert 32768 * 8 * bench._row_bytes("f16", 128) == 134_217_728
    assert 32768 * 8 * bench._row_bytes("q8", 128) == 69_206_016
    assert 32768 * 8 * bench._row_bytes("k8v4", 128) == 53_477_376


def test_step_context_grows_one_cell_per_layer_round():
    L = 32768
    # step s decodes layer s % LAYERS after its append: the context is the
    # prefill plus the cells appended to that layer so far, this one included
    assert bench._step_ctx(0, L) == L + 1
    assert bench._step_ctx(bench.LAYERS - 1, L) == L + 1
    assert bench._step_ctx(bench.LAYERS, L) == L + 2
    # after STEPS_PER_LAYER rounds the workload's cycle starts again
    assert bench._step_ctx(bench.LAYERS * bench.STEPS_PER_LAYER, L) == L + 1


def test_traffic_is_reported_only_for_the_recorded_sources(monkeypatch):
    real = bench._decode_sources_sha()
    f16, q8 = bench._ncu_traffic("f16"), bench._ncu_traffic("q8")
    if f16 is not None:
        # a record taken on the current sources stays within a few percent
        # of the algorithmic bytes of one launch (no re-reads)
        assert 1.0 <= f16 / (32769 * 8 * 512) <= 1.05
        assert 1.0 <= q8 / (32769 * 8 * 264) <= 1.05
    monkeypatch.setattr(bench, "_decode_sources_sha", lambda: "0" * 16)
    assert bench._ncu_traffic("f16") is None      # sources changed: no stale figure
    monkeypatch.setattr(bench, "_decode_sources_sha", lambda: real)
    assert bench._ncu_traffic("f16") == f16
