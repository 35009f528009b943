"""How sensitive the 8B-shaped model's hidden states are to the fp16 rounding
points, measured on the oracle alone (no GPU).

Nudging every 7th weight of the first norm by a factor 1 + 2^-20 (far below any
fp32 arithmetic difference) flips a few fp16 roundings of the normed
activations, and the random-weight network carries the flips to every later
layer.  The oracle's own hidden states then move by more than 1e-3 (relative L2)
at depth while its logits move by far less than 5e-2.  This is why the 1e-3
hidden-state bound is applied layer by layer (each layer fed the same input) and
the end-to-end hidden-state check uses a looser bound.
"""
import numpy as np
import pytest

import oracle
import synth


@pytest.mark.slow
def test_8b_hidden_states_amplify_rounding_flips():
    S = synth.LLAMA3_8B
    w = synth.model_weights(S, 0)
    P = synth.DENSE_8B_CASE["prefill"]
    k, v = synth.kv_prefill(S, 0, 0, P)
    tok = synth.tokens(0, "8b-steps", 8, S.vocab)[:1]

    def run(wd):
        om = oracle.OracleModel(S, wd)
        c = om.new_cache(P + 1, k, v)
        lg, _, h = om.step(tok, [P], [c], P + 1, want_hidden=True)
        return lg[0], h[0]

    lg0, h0 = run(w)
    w2 = dict(w)
    w2["blk.0.attn_norm"] = w["blk.0.attn_norm"].copy()
    w2["blk.0.attn_norm"][::7] *= np.float32(1 + 2.0 ** -20)
    lg1, h1 = run(w2)
    rel = [np.linalg.norm(h1[l] - h0[l]) / np.linalg.norm(h0[l]) for l in range(S.n_layers + 1)]
    assert rel[0] == 0.0
    assert rel[-1] > 1e-3  # end to end, 1e-3 is below the model's own sensitivity
    assert max(rel) < 1e-2
    assert np.abs(lg1 - lg0).max() < 5e-2
