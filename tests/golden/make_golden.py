"""Writes the closed-form fixtures in this folder.

Every value below is derived by hand from the equations cited in each fixture's
"source" field; the derivation is stored beside the numbers. Nothing here calls
the CUDA path (or the oracle): the fixtures pin the oracle from outside.
Run: python tests/golden/make_golden.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def main():
    ln3 = math.log(3.0)
    gate = {
        "source": "TokenGate deep dive (agientry.com), section 3.1, Eq. (3): b~_j = MLP(a~_j); "
                  "read as s = w2 . SiLU(W1 a~_j), g = sigmoid(s), non-prunable tokens carry g = 1",
        "derivation": "W1 = I (2x2), w2 = (1, 1). Row 0: u = (ln 3, 0); SiLU(ln 3) = ln3 * sigmoid(ln3) "
                      "= ln3 * 3/4; SiLU(0) = 0; s = 3/4 ln 3; g = 1/(1 + 3^(-3/4)). Row 1: u = (0, -ln 3); "
                      "SiLU(-ln3) = -ln3 * 1/4; s = -1/4 ln 3; g = 1/(1 + 3^(1/4)). Row 2 is non-prunable: "
                      "same s as row 0, g = 1.",
        "h": [[ln3, 0.0], [0.0, -ln3], [ln3, 0.0]],
        "W1": [[1.0, 0.0], [0.0, 1.0]],
        "w2": [1.0, 1.0],
        "instr_mask": [0, 0, 1],
        "s": [0.75 * ln3, -0.25 * ln3, 0.75 * ln3],
        "g": [1.0 / (1.0 + 3.0 ** -0.75), 1.0 / (1.0 + 3.0 ** 0.25), 1.0],
    }
    att = {
        "source": "TokenGate deep dive (agientry.com), section 3.2, Eq. (5); TokenGate paper page "
                  "(thelatestinai.com), Figure 1 (c): each attention weight is multiplied by its key's "
                  "gate value and renormalised",
        "derivation": "All keys are zero vectors, so every logit q.k/sqrt(d) is 0 and exp(z) = 1. Eq. (5) "
                      "then gives alpha_ij = g_j / sum_{j'<=i} g_j'. With g = (1/2, 1/4, 1/4), beta = 1, "
                      "tau = 1 and V = identity rows, o_0 = (1, 0, 0), o_1 = (2/3, 1/3, 0), "
                      "o_2 = (1/2, 1/4, 1/4).",
        "Q": [[[1.0, 2.0, -1.0]], [[0.5, 0.0, 3.0]], [[-2.0, 1.0, 1.0]]],
        "K": [[[0.0, 0.0, 0.0]], [[0.0, 0.0, 0.0]], [[0.0, 0.0, 0.0]]],
        "V": [[[1.0, 0.0, 0.0]], [[0.0, 1.0, 0.0]], [[0.0, 0.0, 1.0]]],
        "g": [0.5, 0.25, 0.25],
        "tau": [1.0], "beta": [1.0],
        "O": [[[1.0, 0.0, 0.0]], [[2.0 / 3.0, 1.0 / 3.0, 0.0]], [[0.5, 0.25, 0.25]]],
    }
    sel = {
        "source": "TokenGate deep dive (agientry.com), section 3.1, Eq. (4): S = topK over P of b_j, "
                  "union N; section 3.4: the budget is clamped to |P| and the keep indices cover the "
                  "full sequence in original order",
        "derivation": "One sequence of 8 rows; rows 0 and 5 are non-prunable. Document scores by row: "
                      "1:0.5, 2:3.0, 3:-1.0, 4:3.0, 6:0.5, 7:2.0. Ranking by score, ties to the lower row: "
                      "2, 4, 7, 1, 6, 3. K=0 keeps only {0,5}; K=1 adds 2; K=2 adds 4; K=3 adds 7; "
                      "K=4 adds 1; K=5 adds 6; K>=6 keeps all 8 rows.",
        "s": [9.0, 0.5, 3.0, -1.0, 3.0, -7.0, 0.5, 2.0],
        "instr_mask": [1, 0, 0, 0, 0, 1, 0, 0],
        "cu_seqlens": [0, 8],
        "expected": {
            "0": [0, 5], "1": [0, 2, 5], "2": [0, 2, 4, 5], "3": [0, 2, 4, 5, 7],
            "4": [0, 1, 2, 4, 5, 7], "5": [0, 1, 2, 4, 5, 6, 7], "6": [0, 1, 2, 3, 4, 5, 6, 7],
            "9": [0, 1, 2, 3, 4, 5, 6, 7],
        },
    }
    norm = {
        "source": "TokenGate deep dive (agientry.com), section 3.1, Eq. (3): b_j = b~_j / sqrt(mean over P "
                  "of b~^2 + eps), b_j = 0 on N; section 3.2, Eq. (7): tau_i = softplus(sigma) log m_i / "
                  "log max(2, p_i)",
        "derivation": "Two sequences. Sequence 0: raw scores (3, 4, 9) with row 2 non-prunable; mean of squares "
                      "over P = (9 + 16)/2 = 12.5, so b = (3, 4)/sqrt(12.5) = (0.6 sqrt 2, 0.8 sqrt 2) and b_2 = 0. "
                      "Sequence 1: raw scores (-2, 2, 2, -2), all prunable; mean square 4, so b = (-1, 1, 1, -1). "
                      "eps = 0. Temperatures with softplus(sigma) = 1.5: (m, p) = (1, 1) -> 0; (2, 2) -> 1.5; "
                      "(2, 4) -> 1.5 ln 2 / ln 4 = 0.75; (3, 9) -> 1.5 ln 3 / ln 9 = 0.75.",
        "s": [3.0, 4.0, 9.0, -2.0, 2.0, 2.0, -2.0],
        "instr_mask": [0, 0, 1, 0, 0, 0, 0],
        "cu_seqlens": [0, 3, 7],
        "b": [0.6 * math.sqrt(2.0), 0.8 * math.sqrt(2.0), 0.0, -1.0, 1.0, 1.0, -1.0],
        "temp": 1.5,
        "tau_cases": [[1, 1, 0.0], [2, 2, 1.5], [2, 4, 0.75], [3, 9, 0.75]],
    }
    for name, obj in (("gate_score_closed_form.json", gate), ("attention_zero_logits.json", att),
                      ("select_worked_example.json", sel), ("normalized_scores_closed_form.json", norm)):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(obj, f, indent=1)


if __name__ == "__main__":
    main()
