"""The single-GPU price table (the per-bucket slice of the Zellige paper's
Hardware Profiler, arXiv 2608.01150v1 §IV-B) and its additive model."""
import math

import pytest

from mixed_length_dit_gb300 import profiler


def test_catalog_matches_paper_token_counts():
    names = {b.name: b.tokens for b in profiler.catalog()}
    # §I: a 15-second 1080p video is 497,760 tokens; Fig. 1: a 256p image is 256
    assert names["vid_1080p_15s"] == 497760
    assert names["img_256p"] == 256
    # Fig. 2: a 720p 10-second video is 41 x 45 x 80 tokens, a 720p image 45 x 80
    assert names["vid_720p_10s"] == 41 * 45 * 80
    assert names["img_720p"] == 45 * 80
    toks = [b.tokens for b in profiler.catalog()]
    assert toks == sorted(toks)


def test_additive_prediction():
    bks = [profiler.Bucket("a", 1000, "image"), profiler.Bucket("b", 4000, "video")]
    prices = {"a": 1.0, "b": 10.0}
    assert profiler.predict_ms([1000, 1000, 4000], prices, bks) == pytest.approx(12.0)
    # a length between buckets takes the nearest one, scaled quadratically
    assert profiler.predict_ms([2000], prices, bks) == pytest.approx(1.0 * 4)
    assert profiler.predict_ms([0, 3000], prices, bks) == pytest.approx(10.0 * (3000 / 4000) ** 2)
    with pytest.raises(ValueError):
        profiler.predict_ms([10], {}, bks)


@pytest.mark.gpu
def test_prices_predict_a_mixed_batch():
    """Prices measured per bucket predict the time of a coalesced mixed batch
    of those buckets (the additive model the paper evaluates in §V-B)."""
    bks = [b for b in profiler.catalog() if b.name in ("img_480p", "img_1080p", "vid_480p_5s", "vid_720p_5s")]
    prices = profiler.measure_prices(bks, num_heads=12, fill_tokens=200_000, reps=3)
    for b in bks:
        assert prices[b.name] > 0
    # quadratic work: a longer bucket costs more per sequence
    by = sorted(bks, key=lambda b: b.tokens)
    assert all(prices[x.name] < prices[y.name] for x, y in zip(by, by[1:]))
    mix = [b.tokens for b in bks for _ in range(6)]
    measured = profiler.time_batch(mix, num_heads=12)
    predicted = profiler.predict_ms(mix, prices, bks)
    assert abs(predicted - measured) / measured < 0.25, (predicted, measured)


def test_lpt_estimate_equals_additive_when_items_fill_the_sms():
    """Many equal items per SM: the schedule replay gives the sum of prices."""
    bks = [profiler.Bucket("a", 1024, "image")]
    prices = {"a": 2.0}
    seqs = [1024] * (152 * 2)          # 4 forward items per head x 2 heads each, 32 backward per head
    lpt = profiler.predict_lpt_ms(seqs, prices, bks, num_heads=2, head_dim=128, sms=152)
    assert lpt == pytest.approx(profiler.predict_ms(seqs, prices, bks), rel=1e-9)
    assert profiler.predict_lpt_ms(seqs, prices, bks, 2, 128, sms=152, mode="fwd") == \
        pytest.approx(profiler.predict_ms(seqs, prices, bks), rel=1e-9)
    # a measured forward price splits the sequence's time between the launches
    lpt_f = profiler.predict_lpt_ms(seqs, prices, bks, 2, 128, sms=152, fwd_prices={"a": 0.5})
    assert lpt_f == pytest.approx(profiler.predict_ms(seqs, prices, bks), rel=1e-9)


def test_lpt_estimate_shows_the_tail_of_few_items():
    """One sequence with fewer items than SMs takes as long as its longest
    item, not its share of the GPU."""
    bks = [profiler.Bucket("a", 1024, "image")]
    prices = {"a": 1.0}
    one = profiler.predict_lpt_ms([1024], prices, bks, num_heads=1, head_dim=128, sms=152, mode="fwd")
    # 4 equal forward items: each holds an SM for 152/4 of the price
    assert one == pytest.approx(152 / 4)
    more = profiler.predict_lpt_ms([1024, 256], prices, bks, num_heads=1, head_dim=128, sms=152, mode="fwd")
    assert more >= one
    with pytest.raises(ValueError):
        profiler.predict_lpt_ms([10], {}, bks, num_heads=1, sms=152)


def test_lpt_estimate_with_a_tile_table():
    """A split sequence's forward items come from its tiles; its price is the
    whole sequence's, spread over the tiles' items by their work.  A 2 x 2
    grid of one 2,048-token sequence on one head: 16 forward items (four
    query blocks of 256 rows in each of the 4 tiles of 1,024 x 1,024) of
    equal work."""
    import synth
    bks = [profiler.Bucket("a", 2048, "video")]
    tiles = synth.grid_tiles(0, 2048, 2048, 2, 2)
    one = profiler.predict_lpt_ms([2048], {"a": 1.0}, bks, num_heads=1, head_dim=128, sms=152, mode="fwd",
                                  tiles=tiles)
    assert one == pytest.approx(152 / 16)


@pytest.mark.gpu
@pytest.mark.parametrize("n", [3, 5, 7])
def test_schedule_replay_predicts_measured_batches(n):
    """Prices measured on this GPU for the batch's own sequence lengths,
    replayed through the launch's schedule, predict the measured fwd+bwd time
    of the mixed Wan batch (3), the training-step batch with its 2 x 2 split
    video (5) and the Fig. 2 batch of three split 720p videos and 228 images
    (7) within 10% (the paper's profiler reports a makespan error of a few
    percent, §V-B)."""
    import synth
    wl = synth.config(n)
    r = profiler.validate_batch(wl.seqlens, wl.num_heads, wl.head_dim, tiles=wl.tiles() or None)
    assert r["measured_ms"] > 0
    assert abs(r["lpt_err"]) <= 0.10, r
