"""The chunked-prefill step budget, restated (oracle, test-only).

"How LLM Inference Serving Works", section "Chunked prefill": every step has a
token budget; the scheduler takes all pending decode requests first (one token
each), and any remaining budget goes to pending prefills in order; a prefill
that does not fit is cut to what is left ("chunked").  Readings where the page
is silent: more decodes than the budget -> the first ``budget`` decodes run and
no prefill does; prefills are served strictly in queue order, each taking
min(its remaining tokens, budget left), so at most the last one scheduled is
cut.
"""


def plan_step(budget, num_decodes, prefill_remaining):
    """Returns (decodes scheduled, [tokens scheduled per pending prefill])."""
    if budget < 0 or num_decodes < 0 or any(r < 0 for r in prefill_remaining):
        raise ValueError("negative input")
    decodes = min(num_decodes, budget)
    left = budget - decodes
    chunks = []
    for r in prefill_remaining:
        take = min(r, left)
        chunks.append(take)
        left -= take
    return decodes, chunks
