"""CPU pins of the oracle's greedy self-speculative loop and its toy model.

The loop ([PTI-readme] "打包双子推理（PTI）" §"接受机制如何工作"; state handling of
[PTI-forum] §"技术实现架构") is pinned against a plain greedy rollout (the text
it confirms must be exactly the model's greedy continuation: the pages' "zero
quality loss"), against closed forms of planted next-token tables (a fixed
point, a successor chain) and against its bounds; the toy model's logits
against a direct composition of the already-pinned layer and GEMV.
"""
import numpy as np
import pytest

import oracle
import pti_synth


def rollout(nxt, first, count):
    out, t = [], first
    for _ in range(count):
        t = int(nxt[t])
        out.append(t)
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("n", [1, 2, 3, 4])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_confirmed_text_is_the_greedy_rollout(n, seed):
    rng = np.random.default_rng(seed)
    vocab = 37
    # a random table, with some short cycles and fixed points planted
    nxt = rng.integers(0, vocab, vocab).astype(np.int32)
    nxt[5] = 5
    nxt[7], nxt[8] = 8, 7
    for first in range(vocab):
        tokens, accept = oracle.selfspec_greedy(nxt, n, first, 30)
        assert tokens.size == int(np.sum(accept)) + 30
        assert np.all((accept >= 0) & (accept <= n - 1))
        np.testing.assert_array_equal(tokens, rollout(nxt, first, tokens.size))


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_fixed_point_accepts_every_guess_after_the_first_step(n):
    vocab, star = 16, 3
    nxt = np.full(vocab, star, dtype=np.int32)  # every token leads to the fixed point 3
    steps = 9
    tokens, accept = oracle.selfspec_greedy(nxt, n, 11, steps)
    # step 0: the window holds 11 everywhere, every stream outputs 3, the guess
    # 11 of stream 1 is wrong: one token; from then on the window is all 3
    np.testing.assert_array_equal(accept, [0] + [n - 1] * (steps - 1))
    assert tokens.size == 1 + (steps - 1) * n
    assert np.all(tokens == star)
    # starting on the fixed point itself, every step confirms n tokens
    tokens, accept = oracle.selfspec_greedy(nxt, n, star, steps)
    np.testing.assert_array_equal(accept, [n - 1] * steps)
    assert tokens.size == steps * n


@pytest.mark.parametrize("n", [2, 3, 4])
def test_successor_chain_confirms_one_token_per_step(n):
    # next(t) = t + 1 mod V has no fixed point; every stream of the window gets
    # the same token after the first step, so stream 1's guess is always its
    # own input and never the model's next token: one token per step
    vocab = 50
    nxt = ((np.arange(vocab) + 1) % vocab).astype(np.int32)
    tokens, accept = oracle.selfspec_greedy(nxt, n, 4, 20)
    assert np.all(accept == 0)
    np.testing.assert_array_equal(tokens, (np.arange(5, 25) % vocab).astype(np.int32))


def test_two_cycle_and_hand_traced_window():
    # next: 0 -> 1 -> 2 -> 1 (a 2-cycle {1, 2} entered from 0); n = 3
    nxt = np.array([1, 2, 1], dtype=np.int32)
    tokens, accept = oracle.selfspec_greedy(nxt, 3, 0, 3)
    # step 0: win (0,0,0) -> a (1,1,1); win[1]=0 != 1: L=0, confirm 1, win (1,1,1)
    # step 1: a (2,2,2); win[1]=1 != 2: L=0, confirm 2, win (2,2,2)
    # step 2: a (1,1,1); win[1]=2 != 1: L=0, confirm 1
    np.testing.assert_array_equal(tokens, [1, 2, 1])
    np.testing.assert_array_equal(accept, [0, 0, 0])


def test_bad_arguments_are_rejected():
    nxt = np.array([1, 0], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.selfspec_greedy(nxt, 5, 0, 1)
    with pytest.raises(ValueError):
        oracle.selfspec_greedy(nxt, 2, 2, 1)
    with pytest.raises(ValueError):
        oracle.selfspec_greedy(np.array([1, 2], dtype=np.int32), 2, 0, 1)


def test_greedy_next_table_takes_the_lowest_index_on_ties():
    lg = np.array([[0.0, 2.0, 2.0], [5.0, -1.0, 4.0], [1.0, 1.0, 1.0]])
    nxt, margin = oracle.greedy_next_table(lg)
    np.testing.assert_array_equal(nxt, [1, 0, 0])
    np.testing.assert_allclose(margin, [0.0, 1.0, 0.0])


def test_toy_logits_compose_the_pinned_layer_and_gemv():
    m = pti_synth.toy_model(64, 256, 256, seed=3)
    toks = np.array([0, 17, 63, 17])
    lg = oracle.toy_logits(m["embedding"], m["w_gate"], m["w_up"], m["w_down"], m["w_head"],
                           64, 256, 256, toks)
    assert lg.shape == (4, 64)
    np.testing.assert_array_equal(lg[1], lg[3])  # the logits depend on the token only
    # direct composition: embedding row -> fp64 layer -> fp32-rounded output
    # through the fp32 GEMV; the fp64 head differs from it by at most the
    # GEMV's rounding of the layer output (2^-24 relative per element)
    x = m["embedding"][toks]
    xo, _ = oracle.mlp_layer(m["w_gate"], m["w_up"], m["w_down"], 256, 256, x)
    y32, bound = oracle.q8_gemv(m["w_head"], 64, 256, xo.astype(np.float32))
    assert np.all(np.abs(lg - y32) <= 2.0 ** -23 * bound + 1e-300)
