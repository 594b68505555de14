"""Writes the hand-worked fixtures in this folder.

The pages print no worked numeric example, so every value here is a closed
form derived by hand from the definitions (the derivation is stored beside the
numbers).  This script uses only ``math``; it calls neither the oracle nor the
CUDA path.  Run: python tests/golden/make_hand_fixtures.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = "DeepSeek-V3.2 32k long-sequence pretraining on Ascend page, section SparseLightningIndexerGradKLLoss"


def dump(name, obj):
    with open(os.path.join(HERE, name), "w") as f:
        json.dump(obj, f, indent=1)


def main():
    dump("indexer_hand.json", {
        "cite": SRC + ": Lightning Indexer forward formula I[t,:] = W[t,:] ReLU(q~[t] K~^T), causal keys s <= pos(t)",
        "derivation": [
            "one query token at global position 1, two index heads, d_I = 2",
            "s=0: head0 q.k = 1*1+2*0 = 1 -> relu 1; head1 = -1*1+1*0 = -1 -> relu 0; I = 0.5*1 + 2*0 = 0.5",
            "s=1: head0 = 1*0+2*1 = 2; head1 = -1*0+1*1 = 1; I = 0.5*2 + 2*1 = 3",
            "s=2: not visible from position 1 -> -inf"],
        "q_I": [[[[1.0, 2.0], [-1.0, 1.0]]]],
        "k_I": [[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]],
        "w": [[[0.5, 2.0]]],
        "pos": [[1]],
        "expected_I": [[[0.5, 3.0, None]]],
    })

    dump("topk_hand.json", {
        "cite": SRC + ": top-k positions of each token (the order rule -- ties to the lower index, -0 == +0, "
                      "ascending output, -1 padding -- is this library's stated reading)",
        "scores": [1.0, 3.0, -0.0, 3.0, 0.0, 2.0, 3.0],
        "cases": [
            {"pos": 6, "k": 2, "expected": [1, 3], "why": "three 3.0s tie; the two lower indices win"},
            {"pos": 6, "k": 3, "expected": [1, 3, 6], "why": "all three 3.0s"},
            {"pos": 6, "k": 5, "expected": [0, 1, 3, 5, 6], "why": "3,3,3,2,1"},
            {"pos": 6, "k": 6, "expected": [0, 1, 2, 3, 5, 6], "why": "-0.0 at 2 equals 0.0 at 4; lower index 2 wins"},
            {"pos": 3, "k": 2, "expected": [1, 3], "why": "only keys 0..3 visible"},
            {"pos": 6, "k": 9, "expected": [0, 1, 2, 3, 4, 5, 6, -1, -1], "why": "k above the 7 visible keys: all, then -1"},
            {"pos": 0, "k": 3, "expected": [0, -1, -1], "why": "the first token sees only itself"},
        ],
    })

    ln3 = math.log(3.0)
    kv = [[1.0, 2.0, 0.0], [9.0, 9.0, 9.0], [3.0, 4.0, ln3]]
    dump("attention_hand.json", {
        "cite": SRC + ": Sparse Flash Attention forward p = Softmax(q K_topk^T / sqrt(d)); V = first d_v columns "
                      "of the shared kv row (weight absorption)",
        "derivation": [
            "scale 1, H = 2, d_qk = 3, d_v = 2; the token selects keys 0 and 2 (third slot is -1 padding)",
            "head0 q = [0,0,1]: logits [kv0[2], kv2[2]] = [0, ln 3]; m = ln 3; exp(s-m) = [1/3, 1]; l = 4/3; P = [1/4, 3/4]",
            "O(head0) = 1/4*[1,2] + 3/4*[3,4] = [2.5, 3.5]",
            "head1 q = 0: logits [0,0]; m = 0; l = 2; P = [1/2,1/2]; O(head1) = [2, 3]",
            "kv row 1 = [9,9,9] is not selected and must not contribute"],
        "scale": 1.0, "d_v": 2,
        "q": [[[[0.0, 0.0, 1.0], [0.0, 0.0, 0.0]]]],
        "kv": [kv],
        "idx": [[[0, 2, -1]]],
        "expected_O": [[[[2.5, 3.5], [2.0, 3.0]]]],
        "expected_m": [[[ln3, 0.0]]],
        "expected_l": [[[4.0 / 3.0, 2.0]]],
    })

    e3 = math.exp(1.0), math.exp(3.0)
    pi0, pi1 = e3[0] / (e3[0] + e3[1]), e3[1] / (e3[0] + e3[1])
    p0, p1 = 0.25, 0.75
    loss = p0 * math.log(p0 / pi0) + p1 * math.log(p1 / pi1)
    dI0, dI1 = pi0 - p0, pi1 - p1
    dump("kl_loss_hand.json", {
        "cite": SRC + ": Loss = sum_t KL(p_t || Softmax(I_t)); dI = Softmax(I) - p; dW = dI ReLU(S)^T; "
                      "dq~ = dS K~_topk; dK~_topk = dS^T q~",
        "derivation": [
            "attention part: H = 1, scale 1, q = [0,0,1]; selected keys 0 and 2 with logits 0 and ln 3 -> "
            "P = [1/4, 3/4] = p (one head, already L1-normalised)",
            "indexer: H_I = 1, d_I = 1, q~ = 1, k~ = [1, 5, 3], w = 1: S = [1, 3] on keys 0, 2 -> I = [1, 3], "
            "pi = softmax(I) = [e/(e+e^3), e^3/(e+e^3)]",
            "loss = 1/4 ln((1/4)/pi0) + 3/4 ln((3/4)/pi1)",
            "dI = [pi0 - 1/4, pi1 - 3/4]; dw = dI0*1 + dI1*3; dq~ = w*(dI0*1 + dI1*3); "
            "dk~[0] = dI0*w*q~, dk~[2] = dI1*w*q~, dk~[1] = 0 (not selected)"],
        "scale": 1.0,
        "q": [[[[0.0, 0.0, 1.0]]]],
        "kv": [kv],
        "idx": [[[0, 2]]],
        "m": [[[ln3]]], "l": [[[4.0 / 3.0]]],
        "q_I": [[[[1.0]]]], "k_I": [[[1.0], [5.0], [3.0]]], "w": [[[1.0]]],
        "expected_loss": loss,
        "expected_dw": [[[dI0 + 3 * dI1]]],
        "expected_dq_I": [[[[dI0 + 3 * dI1]]]],
        "expected_dk_I": [[[dI0], [0.0], [dI1]]],
    })

    # Two attention heads whose softmax sums l differ, so the target p depends
    # on normalising each head by its own l before the head sum.
    q0, q1 = 3.0 / 8.0, 5.0 / 8.0
    loss2 = q0 * math.log(q0 / pi0) + q1 * math.log(q1 / pi1)
    dJ0, dJ1 = pi0 - q0, pi1 - q1
    dump("kl_loss_hand_2heads.json", {
        "cite": SRC + ": the target p sums the attention probabilities over all heads, then L1-normalises "
                      "along the context; Loss = sum_t KL(p_t || Softmax(I_t)); dI = Softmax(I) - p",
        "derivation": [
            "attention part: H = 2, scale 1, selected keys 0 and 2 of the kv rows below",
            "head 0: q = [0,0,1] -> logits [0, ln 3]; m = ln 3, l = 4/3; P = [1/4, 3/4]",
            "head 1: q = [0,0,0] -> logits [0, 0]; m = 0, l = 2; P = [1/2, 1/2]",
            "head sum [3/4, 5/4] over the total 2 -> p = [3/8, 5/8]",
            "(without the per-head division by l the head sum of exp(s - m) is [4/3, 2] and p would be "
            "[2/5, 3/5]; weighting heads by l gives yet another p)",
            "indexer part as in kl_loss_hand.json: I = [1, 3] on keys 0, 2, pi = softmax(I)",
            "loss = 3/8 ln((3/8)/pi0) + 5/8 ln((5/8)/pi1); dI = [pi0 - 3/8, pi1 - 5/8]",
            "dw = dI0*1 + dI1*3; dq~ = dI0*1 + dI1*3; dk~[0] = dI0, dk~[2] = dI1, dk~[1] = 0"],
        "scale": 1.0,
        "q": [[[[0.0, 0.0, 1.0], [0.0, 0.0, 0.0]]]],
        "kv": [kv],
        "idx": [[[0, 2]]],
        "m": [[[ln3, 0.0]]], "l": [[[4.0 / 3.0, 2.0]]],
        "q_I": [[[[1.0]]]], "k_I": [[[1.0], [5.0], [3.0]]], "w": [[[1.0]]],
        "expected_p": [q0, q1],
        "expected_loss": loss2,
        "expected_dw": [[[dJ0 + 3 * dJ1]]],
        "expected_dq_I": [[[[dJ0 + 3 * dJ1]]]],
        "expected_dk_I": [[[dJ0], [0.0], [dJ1]]],
    })


if __name__ == "__main__":
    main()
