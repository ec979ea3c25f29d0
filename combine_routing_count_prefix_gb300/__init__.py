"""GB300-native low-latency MoE dispatch / combine (one GPU, R simulated ranks).

Submodules:

- ``llmoe``: the Python binding of the C-ABI library ``libllmoe.so``
  (``llmoe_layout_bytes``, ``llmoe_dispatch``, ``llmoe_combine``,
  ``llmoe_clean``, ...).  Importing it loads the library and raises if it has
  not been built: there is no fallback path.
- ``build``: compiles the CUDA library for sm_103a.
- ``inputs``: seeded synthetic workloads.
"""
