"""Writes the closed-form fixtures in this folder (no oracle, no GPU).

hand_example.json: a 2-row, H=2, V=3 problem solved by hand from the
definition (logits = h W^T; per-row log-softmax cross entropy against the
label; label -100 ignored; mean over the rest). The numbers are the hand
derivation evaluated with the math module.

w_zero.json: with W = 0 every logit is 0, so log-sum-exp = ln V exactly.

Run: python tests/golden/make_closed_forms.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    e = math.e
    d = e + 2.0
    hand = {
        "description": "Worked example derived by hand from the definition: "
                       "logits = h W^T, per-row log-softmax cross entropy "
                       "against the label, rows with label -100 ignored, "
                       "mean over the remaining rows.",
        "source": "Training Beyond 1M Tokens (TRL guide), section 'The loss "
                  "is the first thing to break' (logits L x V = hidden L x H "
                  "times LM-head weights, cross entropy against target "
                  "labels); reduction and ignore_index are this library's "
                  "reading of what the pages leave open",
        "derivation": [
            "row 0: z = [1, 0, 0], lse = ln(e + 2), label 0 -> loss term ln(e + 2) - 1",
            "row 1: z = [0, 2, 0], lse = ln(2 + e^2), label -100 -> ignored, N = 1",
            "loss = ln(e + 2) - 1",
            "softmax row 0 = [e, 1, 1] / (e + 2); G row 0 = softmax - onehot(0) = [-2, 1, 1] / (e + 2); G row 1 = 0",
            "dH = G W = [[-2/(e+2), 1/(e+2)], [0, 0]]",
            "dW = G^T h = [[-2/(e+2), 0], [1/(e+2), 0], [1/(e+2), 0]]",
        ],
        "h": [[1.0, 0.0], [0.0, 2.0]],
        "W": [[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]],
        "labels": [0, -100],
        "dloss": 1.0,
        "expected": {
            "lse": [math.log(d), math.log(2.0 + e * e)],
            "loss": math.log(d) - 1.0,
            "n_valid": 1,
            "dH": [[-2.0 / d, 1.0 / d], [0.0, 0.0]],
            "dW": [[-2.0 / d, 0.0], [1.0 / d, 0.0], [1.0 / d, 0.0]],
        },
    }
    with open(os.path.join(HERE, "hand_example.json"), "w") as f:
        json.dump(hand, f, indent=1)
    wz = {
        "description": "Closed form at W = 0: every logit is 0, so every "
                       "row's log-sum-exp is ln V, the loss is ln V whatever "
                       "the labels, dH = 0 and dW[v] = (dloss/N) * sum over "
                       "valid rows of (1/V - [y_i = v]) h_i.",
        "source": "Follows from the definition in Training Beyond 1M Tokens "
                  "(TRL guide), section 'The loss is the first thing to "
                  "break'; V = 151936 is the Qwen3 vocabulary of the head "
                  "shapes, V = 4096 the small case",
        "ln_V": {"4096": math.log(4096), "151936": math.log(151936)},
    }
    with open(os.path.join(HERE, "w_zero.json"), "w") as f:
        json.dump(wz, f, indent=1)


if __name__ == "__main__":
    main()
