"""GB300-native hot path of stochastic dynamic-tree speculative decoding.

The compute path is the C-ABI library libspec_tree.so (include/spec_tree.h),
reached from Python through `dynamic_tree_speculative_gb300.binding`.
`workloads` holds the seeded synthetic input generators.
"""
__all__ = ["binding", "workloads"]
