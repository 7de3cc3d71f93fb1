"""Writes closed_form_cases.json: two attention problems solved by hand.

The values below come from the definition of scaled dot-product attention
(softmax of the scaled scores, natural-log log-sum-exp per row, top-left
causal mask) and its derivative, worked out on paper; this script only
evaluates the resulting closed forms (ln 2, ln 3, sqrt 2) to float64 and
calls neither the oracle nor the library. Run it from the repository root.
"""

import json
import math

ln2, ln3, s2 = math.log(2), math.log(3), math.sqrt(2)

CASES = {
    "citation": (
        "Definition of scaled dot-product attention, out = softmax(scale*Q K^T + causal) V with "
        "the natural-log log-sum-exp of each score row stashed for the backward "
        "('Scaled_dot_product_attention', discuss.pytorch.org thread; 'DID loop split for SDPA', "
        "NVIDIA/Fuser PR 3711, test_sdpa_loop_split signatures of sdpfa_fwd / sdpfa_bwd). The pages "
        "print no numeric example; these two cases are derived by hand from that definition and its "
        "derivative (dV = P^T dO, dS = P*(dO V^T - rowsum(dO*out)), dQ = scale dS K, "
        "dK = scale dS^T Q), chosen so every softmax weight is a simple fraction."),
    "cases": [
        {"name": "one_query_two_keys",
         "derivation": ("S = [0, ln 3] so P = [1/4, 3/4]; out = 4/4 + 3*8/4 = 7; lse = ln 4. "
                        "dP = [4, 8], Delta = 7, dS = [-3/4, 3/4]; dq = 3/4 * k1 = 3/4; "
                        "dk = dS * q = [-3/4 ln3, 3/4 ln3]; dv = P = [1/4, 3/4]."),
         "is_causal": False, "scale": 1.0,
         "q": [[ln3]], "k": [[0.0], [1.0]], "v": [[4.0], [8.0]], "dout": [[1.0]],
         "out": [[7.0]], "lse": [math.log(4)],
         "dq": [[0.75]], "dk": [[-0.75 * ln3], [0.75 * ln3]], "dv": [[0.25], [0.75]]},
        {"name": "causal_two_by_two",
         "derivation": ("scale = 1/sqrt 2. Row 0 sees key 0 only: S00 = 0, lse0 = 0, out0 = v0 = [3,0]. "
                        "Row 1: S10 = 0, S11 = ln 2, P1 = [1/3, 2/3], lse1 = ln 3, out1 = [1, 4]. "
                        "With dO = I: dS0 = [0, 0]; dP1 = [0, 6], Delta1 = 4, dS1 = [-4/3, 4/3]. "
                        "dQ1 = scale*4/3*(k1-k0) = [2 sqrt2/3, 0]; dK0 = scale*(-4/3)*q1 = [-4/3 ln2, 0]; "
                        "dK1 = [4/3 ln2, 0]; dV0 = [1, 1/3], dV1 = [0, 2/3]."),
         "is_causal": True, "scale": 1.0 / s2,
         "q": [[1.0, 1.0], [s2 * ln2, 0.0]], "k": [[0.0, 0.0], [1.0, 0.0]],
         "v": [[3.0, 0.0], [0.0, 6.0]], "dout": [[1.0, 0.0], [0.0, 1.0]],
         "out": [[3.0, 0.0], [1.0, 4.0]], "lse": [0.0, ln3],
         "dq": [[0.0, 0.0], [2 * s2 / 3, 0.0]], "dk": [[-4 / 3 * ln2, 0.0], [4 / 3 * ln2, 0.0]],
         "dv": [[1.0, 1 / 3], [0.0, 2 / 3]]},
    ],
}

if __name__ == "__main__":
    with open("tests/golden/closed_form_cases.json", "w") as f:
        json.dump(CASES, f, indent=1)
