"""Pins of the loop's slot scheduling (oracle.loop.serve), by closed forms.

* every iteration yields 17 tokens per request (a perfect drafter): a
  request with budget m holds its slot for ceil(m / 17) iterations, so with
  one slot the admission iterations are the running sums of those;
* one token per iteration (drafts never accepted): ceil(m / 1) = m;
* two slots, equal budgets: requests pair up in queue order (slot 0 gets
  the even ones, slot 1 the odd ones) and each pair is admitted together;
* no token is lost or repeated: a request's output is exactly the tokens
  its steps produced, in order;
* requests beyond the iteration count are never admitted.
"""
import math

from oracle.loop import serve


def _const_step(n):
    counter = {}

    def step(active):
        out = {}
        for b, q in active:
            c = counter.get(q, 0)
            out[b] = [1000 * q + c + i for i in range(n)]
            counter[q] = c + n
        return out
    return step


def test_perfect_drafter_one_slot():
    budgets = [5, 40, 17, 18, 1]
    out, admit, gen = serve(budgets, 1, _const_step(17), 20)
    want, t = [], 0
    for m in budgets:
        want.append(t)
        t += math.ceil(m / 17)
    assert admit == want
    assert all(g >= m for g, m in zip(gen, budgets))


def test_one_token_per_iteration():
    budgets = [3, 2, 4]
    out, admit, gen = serve(budgets, 1, _const_step(1), 20)
    assert admit == [0, 3, 5]
    assert gen == budgets


def test_two_slots_pair_up():
    budgets = [4] * 6
    out, admit, gen = serve(budgets, 2, _const_step(1), 30)
    assert admit == [0, 0, 4, 4, 8, 8]


def test_outputs_are_the_steps_tokens_in_order():
    budgets = [7, 3, 9]
    out, admit, gen = serve(budgets, 2, _const_step(2), 30)
    for q, o in enumerate(out):
        assert o == [1000 * q + i for i in range(len(o))]
        assert len(o) == 2 * math.ceil(budgets[q] / 2)


def test_unadmitted_requests():
    out, admit, gen = serve([10, 10, 10], 1, _const_step(1), 12)
    assert admit == [0, 10, -1] and gen[2] == 0
