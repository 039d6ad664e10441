"""GB300-native chunkwise gated delta rule (GDN) / DeltaProduct forward and
camera-branch prep.

The compute path is the C-ABI library ``libgdn.so`` built from ``csrc/`` for
sm_103a; ``binding`` marshals torch tensors into its entry points.  Importing
the package does not load the library: ``binding`` does, and raises if it is
missing.
"""
__all__ = ["binding", "inputs"]
