"""GB300-native speculative-decoding verification (tree mask, greedy and rejection-sampling
acceptance) behind a C ABI (``include/spec_verify.h``).

``import speculative_decoding_tree_mask_gb300`` loads nothing; ``binding`` opens the CUDA
library on first use and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
