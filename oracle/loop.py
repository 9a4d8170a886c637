"""Float64-side model of the device-resident speculative loop (slot scheduling).

TEST INFRASTRUCTURE: part of the CPU oracle (see oracle/__init__.py).

What is followed: the serving loop of continuous batching -- requests that
have finished leave the running batch and waiting requests take the free
places, first come first served ("LLM inference acceleration", section
three, the batching scheduler); each iteration drafts a block per running
request, verifies it with one target pass and appends the accepted tokens
("The Inference Stack Behind OCRia", speculative-decoding section;
HunyuanOCR-1.5 summary, section one, inference steps 1-5).
Readings (the pages give no more): a request leaves its slot once it has
generated at least its budget of tokens; before every iteration the slots
are scanned in order 0..B-1, and each empty slot (or one whose request just
left) takes the next queued request.
"""
from __future__ import annotations


def serve(budgets, slots: int, step, n_iters: int):
    """Run the loop for n_iters iterations.

    budgets: tokens to generate per queued request, in queue order.
    step(active): active = list of (slot, request) for the busy slots; returns
        {slot: list of tokens generated this iteration} (1..17 tokens each).
    Returns (outputs per request, admission iteration per request (-1 never),
    generated count per request).
    """
    q_total = len(budgets)
    slot_req = [-1] * slots
    head = 0
    out = [[] for _ in range(q_total)]
    admit = [-1] * q_total
    for it in range(n_iters):
        for b in range(slots):
            q = slot_req[b]
            if q >= 0 and len(out[q]) >= budgets[q]:
                q = -1
            if q < 0 and head < q_total:
                q = head
                head += 1
                admit[q] = it
            slot_req[b] = q
        active = [(b, q) for b, q in enumerate(slot_req) if q >= 0]
        if not active:
            continue
        got = step(active)
        for b, q in active:
            out[q].extend(got[b])
    return out, admit, [len(o) for o in out]
