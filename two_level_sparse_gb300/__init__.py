"""GB300 (sm_103a) two-level candidate sparse-attention indexer.

``two_level_sparse_gb300.ci`` binds the C ABI of ``libci.so`` (declared in
``include/ci.h``); ``two_level_sparse_gb300.synth`` draws seeded synthetic
inputs.  Importing the package itself loads nothing.
"""
