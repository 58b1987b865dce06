"""The benchmark's roofline arithmetic against the figures derived by hand for the pages'
workloads (per-request byte sums and per-token flop counts), and the headline line's
static parts.  No GPU."""
import bench


def test_decode_bytes_of_the_kimi_shard_layer():
    # per request-layer: S 2*12*128*128*2 = 786,432; window 2*3*4608*2 = 55,296; qkv 9,216;
    # g 6,144; beta 48; o 3,072; slot id 4 -> 860,212; 64 requests + taps 4608*16 = 73,728
    assert bench.decode_bytes_per_launch(1, 12, 128, 128, 2, 2) - 4608 * 16 == 860_212
    assert bench.decode_bytes_per_launch(64, 12, 128, 128, 2, 2) == 64 * 860_212 + 73_728
    assert bench.decode_bytes_per_launch(64, 12, 128, 128, 2, 2) == 55_127_296


def test_decode_bytes_of_the_gdn_layer():
    # fp32 state, bf16 io, gate per head: S 2*32*16384*4 = 4,194,304; window 2*3*12288*2 =
    # 147,456; qkv 24,576; g 128; beta 128; o 8,192; slot id 4 -> 4,374,788 per request
    per_req = 4_194_304 + 147_456 + 24_576 + 128 + 128 + 8_192 + 4
    assert bench.decode_bytes_per_launch(256, 32, 128, 128, 4, 2, per_channel_gate=False) == \
        256 * per_req + 12288 * 16


def test_prefill_flops_of_the_13600_token_prompt():
    assert bench.prefill_flops(1, 1, 128, 128) == 180_224
    assert bench.prefill_flops(13600, 12, 128, 128) == 29_412_556_800


def test_spec_verify_bytes_per_request():
    # read S 393,216 + 8 x 393,216 written; window 27,648 + 8 x 27,648; per token qkv 9,216,
    # g 6,144, beta 48, o 3,072; slot id 4 -> 3,935,620 (~3.94 MB)
    per_req = 9 * 393_216 + 9 * 27_648 + 8 * (9_216 + 6_144 + 48 + 3_072) + 4
    assert per_req == 3_935_620
    assert bench.spec_verify_bytes(64, 8, 12, 128, 128) == 64 * per_req


def test_traffic_is_keyed_by_the_current_decode_sources():
    # the roofline traffic is reported only for the decode kernel the counters came from
    assert bench.decode_source_hash() in bench.CAPTURED_DECODE_TRAFFIC
    assert all(v > 27_000_000 for v in bench.CAPTURED_DECODE_TRAFFIC.values())


def test_end_to_end_groups_cover_every_layer_once():
    assert bench.e2e_bounds(69) == [0, 2, 6, 14, 30, 46, 62, 67, 69]
    for layers in (1, 2, 7, 8, 9, 16, 48, 69, 100):
        b = bench.e2e_bounds(layers)
        assert b[0] == 0 and b[-1] == layers
        assert all(x < y for x, y in zip(b, b[1:])), (layers, b)
