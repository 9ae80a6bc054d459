"""TokenGate gated-prefill hot path for B300 (sm_103a).

The compute lives in the C-ABI library ``libtokengate.so`` (hand-written CUDA);
``binding`` marshals arguments to it and ``inputs`` makes seeded synthetic data.
"""
__all__ = ["binding", "inputs"]
