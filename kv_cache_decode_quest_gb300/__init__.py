"""GB300 (sm_103a) sparse-decode hot path: Quest page selection, split-K GQA
decode attention over an AttentionView, SnapKV compaction and the H2O step.

The compute lives in ``libsparse_engine.so`` (hand-written CUDA, C ABI in
``include/sparse_engine.h``); ``binding`` marshals torch tensors into it.
"""
__all__ = ["binding", "build", "synth", "workloads"]
