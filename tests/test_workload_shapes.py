"""The workload shapes agree with the byte counts printed on "The Neutrino Engine" page."""
from synth import workloads as wl


def _weights_per_layer(shapes):
    return sum(N * K for N, K in shapes.values())


def test_layer_slab_matches_page():
    # § "The file is not the traffic": each layer's weight slab is 72,351,744 bytes, attention
    # 21.7 % and feed-forward 78.3 % of it. 72,351,744 bytes over the layer's weights is
    # exactly 3 bits per weight for these shapes.
    n = _weights_per_layer(wl.DECODER_8B)
    assert n * 3 // 8 == 72_351_744 and (n * 3) % 8 == 0
    attn = sum(wl.DECODER_8B[p][0] * wl.DECODER_8B[p][1] for p in ("q", "k", "v", "o"))
    assert round(100 * attn / n, 1) == 21.7
    assert round(100 * (n - attn) / n, 1) == 78.3


def test_projection_lane_matches_page():
    # Same section: 2.60 GB of ternary projections over 36 layers (at the page's 3 bits).
    total = wl.DECODER_8B_LAYERS * _weights_per_layer(wl.DECODER_8B) * 3 / 8
    assert round(total / 1e9, 2) == 2.60


def test_vocab_tables_match_page():
    # Same section: two untied int8 tables of 151,936 x 4,096, 1.24 GB together.
    assert (wl.HEAD_V, wl.HEAD_K) == (151_936, 4_096)
    assert round(2 * wl.HEAD_V * wl.HEAD_K / 1e9, 2) == 1.24


def test_kv_heads_match_page():
    # § "At 26K tokens, the cache becomes larger than the model": 36 layers, 8 key-value
    # heads of 128 dimensions, 147,456 bytes per cached position at 16 bits.
    kv_dim = wl.DECODER_8B["k"][0]
    assert kv_dim == wl.DECODER_8B["v"][0] == 8 * 128
    assert wl.DECODER_8B_LAYERS * 2 * kv_dim * 2 == 147_456


def test_algorithmic_bytes():
    # 2 bits per trit + fp32 row scale + int8 activation + fp32 output + fp32 activation scale.
    assert wl.packed_bytes_per_token() == 1_748_976_624
    assert wl.head_bytes() == 623_549_448
