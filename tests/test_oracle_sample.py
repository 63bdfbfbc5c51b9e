"""Pins for the oracle's temperature-T draw (Gumbel-max with position-keyed noise) and for
speculative decoding with drawn choices (CPU)."""
import numpy as np
import pytest
import scipy.special
import scipy.stats

import synth
from oracle import model, sample, step


def test_fmix32_is_a_bijection_with_zero_fixed():
    """The finalizer is invertible (distinct inputs, distinct outputs) and maps 0 to 0."""
    x = np.arange(1 << 20, dtype=np.uint32)
    h = sample.fmix32(x)
    assert int(sample.fmix32(0)) == 0
    assert len(np.unique(h)) == len(x)


def test_uniforms_are_uniform_and_inside_the_open_interval():
    u = np.concatenate([sample.uniforms(7, s, n, 4096) for s in range(3) for n in range(20)]).astype(np.float64)
    assert u.min() > 0.0 and u.max() < 1.0
    assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3
    # neighbouring tokens and neighbouring positions are uncorrelated
    a, b = sample.uniforms(7, 0, 5, 100000), sample.uniforms(7, 0, 6, 100000)
    assert abs(np.corrcoef(a[:-1], a[1:])[0, 1]) < 0.02
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.02


def test_gumbel_noise_has_the_gumbel_law():
    g = np.concatenate([sample.gumbel(11, 0, n, 5000) for n in range(40)]).astype(np.float64)
    assert scipy.stats.kstest(g, "gumbel_r").pvalue > 1e-3
    assert abs(g.mean() - np.euler_gamma) < 0.02


@pytest.mark.parametrize("temperature", [0.5, 1.0, 2.0])
def test_draw_frequencies_follow_softmax_at_temperature(temperature):
    """Gumbel-max: P(draw = v) = softmax(logits / T)_v (chi-square over 30000 positions)."""
    logits = np.array([1.3, 0.2, -0.7, 0.9, -2.0, 0.0])
    p = scipy.special.softmax(logits / temperature)
    n = 30000
    counts = np.bincount([sample.draw(logits, temperature, 5, 1, pos) for pos in range(n)], minlength=len(p))
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert scipy.stats.chi2.sf(chi2, len(p) - 1) > 1e-3, (counts, n * p)


def test_small_temperature_draw_is_the_argmax():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(50, 300)) * 4
    got = [sample.draw(logits[i], 1e-4, 9, 0, i) for i in range(50)]
    assert got == list(model.argmax_lowest(logits))


def test_draws_depend_on_sequence_position_and_seed_only():
    logits = np.zeros(1000)  # a uniform distribution: the draw is the noise's argmax
    a = [sample.draw(logits, 1.0, 1, 0, n) for n in range(64)]
    assert a == [sample.draw(logits, 1.0, 1, 0, n) for n in range(64)]          # reproducible
    assert a != [sample.draw(logits, 1.0, 2, 0, n) for n in range(64)]          # seed
    assert a != [sample.draw(logits, 1.0, 1, 1, n) for n in range(64)]          # sequence
    assert len(set(a)) > 50                                                      # positions


@pytest.mark.slow
def test_speculative_sampling_equals_plain_sampling():
    """Losslessness at temperature 1: with the noise keyed to absolute positions, DFlash +
    DDTree with drawn choices emits exactly the tokens plain sampling from the target emits."""
    tw = synth.target_weights(synth.TOY_TARGET, 1002)
    dw = synth.drafter_weights(synth.TOY_DRAFTER, tw, synth.TOY_TARGET.n_feat, 1002)
    prompt = synth.uniform_ints(1002, "prompt", (48,), 0, 512)
    n_new, B, cap = 40, 8, 48 + 40 + 16 + 8
    choose = sample.sampler(1.0, seed=123)
    ref = step.greedy_generate(tw, prompt, n_new + 8, cap, choose)
    assert ref != step.greedy_generate(tw, prompt, n_new + 8, cap)  # not the greedy output
    g = np.random.default_rng(78)

    def plant(st, logits):
        k = len(st.out)
        out = logits.copy()
        for d in range(logits.shape[0]):
            if k + d < len(ref) and g.random() < 0.8:
                out[d, ref[k + d]] += 12.0
        return out

    got, steps = step.spec_generate(tw, dw, prompt, n_new, B, cap, plant, choose)
    assert got == ref[:n_new]
    assert sum(steps) > n_new // 3, steps
    assert max(steps) >= 2
