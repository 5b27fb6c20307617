"""The default kernel path on the device: for ART, the unit path (one item over
many CTAs) for bf16 calls with fewer items than half the SMs, one CTA per item
otherwise; for the dense twin, the unit path with fewer items than SMs. Both paths
give the oracle's result (the parity tests run every case on both with
ART_UNITS)."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _shape(K, batch, hq, hkv, page, ctx, max_visit):
    return K.make_shape(batch=batch, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, page_size=page,
                        block_size=64, max_pages_per_seq=ctx // page, max_visit=max_visit, num_probe=32,
                        num_pages_total=batch * (ctx // page), dtype=0)


def test_default_path_follows_item_count(monkeypatch):
    import kv_cache_early_gb300 as K
    monkeypatch.delenv("ART_UNITS", raising=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cases = [  # the long-context, Llama-shaped (full and batch 2) and paged (batch 8) workloads
        _shape(K, 4, 28, 4, 64, 131072, 600),
        _shape(K, 16, 32, 8, 64, 32768, 512),
        _shape(K, 2, 32, 8, 64, 32768, 512),
        _shape(K, 8, 32, 8, 16, 8192, 128),
    ]
    for shape in cases:
        ws = K.art_workspace_bytes(shape)
        items = shape.batch * shape.num_kv_heads
        expect = 1 if 2 * items < sms else 0
        assert K.art_decode_path(shape, 2, ws) == expect, (items, sms)
        assert K.art_decode_path(shape, 17, ws) == 0  # patience beyond the longest unit
        assert K.dense_decode_path(shape, ws) == (1 if items < sms else 0), (items, sms)
