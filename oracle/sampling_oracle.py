"""Oracle for sampling-based verification (temperature sampling instead of greedy).

TEST INFRASTRUCTURE ONLY.  Plain, slow CPU reference in float64; only the tests, the smoke check and the
bench's CPU-baseline leg may import it.  It shares no code with the CUDA path.

Source: «如何在单张 RTX 3090 上让 Qwen3.5-27B token 生成速度提升 6 倍» (S5), 补充测试 / 关键突破: verification is
greedy (temperature 0) and sampling-based verification is named as future work; «Qwen3.8-27B 部署技术报告»
(S3) runs every test at temperature 0.  The pages give no acceptance rule, so this oracle takes the plainest
reading, standard speculative sampling, with the multi-candidate rule for token trees:

* the target distribution at node u is p_u = softmax(logits_u / T), T > 0;
* the draft distribution at u, from which u's children were drawn, is q_u (given);
* at u the children are tried in increasing node order: child c with token x is accepted when
  r_c * q_u(x) < p(x) (i.e. with probability min(1, p(x) / q_u(x)) for r_c ~ U[0, 1), given per node;
  a token the target gives probability 0 is never accepted);
  after a rejection p becomes the residual max(0, p - q_u), renormalised (kept as is if it sums to 0);
* the walk descends into the accepted child with p = p_child; when every child of the current node is
  rejected, or the node is a leaf, the bonus token is drawn from the current p by inverse CDF with the
  node's own uniform s_u: the smallest token v with sum_{w <= v} p(w) > s_u * sum(p);
* accept length, path and emitted tokens are reported as in the greedy verify (root counted).
"""
from __future__ import annotations

import numpy as np


def softmax_t(logits, temperature: float) -> np.ndarray:
    z = (np.asarray(logits, dtype=np.float64) - np.max(logits)) / float(temperature)
    e = np.exp(z)
    return e / e.sum()


def inverse_cdf(weights, s: float) -> int:
    """Smallest index v with cumsum(weights)[v] > s * sum(weights); weights are >= 0 with a positive sum."""
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    return int(np.searchsorted(c, s * c[-1], side="right"))


def sampling_accept(q_indptr, parents, draft_tokens, logits, draft_probs, temperature, r_accept, r_sample):
    """Returns (accept_len [B], paths, out_tokens, margins).

    margins: per sequence the smallest relative distance of any decision from its threshold (an acceptance
    test |r q - p| / max(p, r q), or the sampled token's position |cdf - s Z| / Z), so that tests can compare
    only decisions that fp32 arithmetic cannot flip.
    """
    logits = np.asarray(logits, dtype=np.float64)
    draft_probs = np.asarray(draft_probs, dtype=np.float64)
    lens, paths, outs, margins = [], [], [], []
    for b in range(len(q_indptr) - 1):
        lo, hi = int(q_indptr[b]), int(q_indptr[b + 1])
        children = [[] for _ in range(hi - lo)]
        for j in range(1, hi - lo):
            children[int(parents[lo + j])].append(j)
        u = 0
        path, toks, margin = [0], [], np.inf
        p = softmax_t(logits[lo], temperature)
        while True:
            accepted = None
            for c in children[u]:
                x = int(draft_tokens[lo + c])
                lhs, rhs = float(r_accept[lo + c]) * draft_probs[lo + u, x], p[x]
                margin = min(margin, abs(lhs - rhs) / max(lhs, rhs, 1e-300))
                if lhs < rhs:
                    accepted = c
                    break
                res = np.maximum(p - draft_probs[lo + u], 0.0)
                if res.sum() > 0:
                    p = res / res.sum()
            if accepted is None:
                s = float(r_sample[lo + u])
                v = inverse_cdf(p, s)
                cdf = np.cumsum(p)
                lo_edge = cdf[v - 1] if v > 0 else 0.0
                margin = min(margin, abs(cdf[v] - s * cdf[-1]) / cdf[-1], abs(s * cdf[-1] - lo_edge) / cdf[-1])
                toks.append(v)
                break
            path.append(accepted)
            toks.append(int(draft_tokens[lo + accepted]))
            u = accepted
            p = softmax_t(logits[lo + u], temperature)
        lens.append(len(path))
        paths.append(path)
        outs.append(toks)
        margins.append(margin)
    return np.array(lens), paths, outs, np.array(margins)
