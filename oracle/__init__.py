"""CPU oracle for the verify step (test infrastructure; see verify_oracle)."""
from .verify_oracle import (PAGE, H_Q, H_KV, GROUP, HEAD_DIM, SCALE, tree_ancestors, gather_context,
                            attend, verify_attention, argmax_first, root_to_leaf_paths,
                            accept_bruteforce, accept, kv_commit)

__all__ = ["PAGE", "H_Q", "H_KV", "GROUP", "HEAD_DIM", "SCALE", "tree_ancestors", "gather_context",
           "attend", "verify_attention", "argmax_first", "root_to_leaf_paths", "accept_bruteforce",
           "accept", "kv_commit"]
