"""GB300-native fused FGP step on the 3D isotropic TV dual.

The compute path is the C-ABI library ``libtvfgp.so`` built from ``csrc/``
(hand-written sm_103a CUDA); ``fgp_dual_stencil_gb300.tvfgp`` is its thin
Python binding.  ``fgp_dual_stencil_gb300.synth`` draws the seeded synthetic
inputs.  Nothing is imported eagerly, so importing the package does not load
the CUDA library.
"""
__all__ = ["tvfgp", "synth"]
