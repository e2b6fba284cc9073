"""Persistent decode megakernel for GB300 (sm_103a).

``runtime`` binds the C-ABI library ``libmk`` (planner + persistent
interpreter kernel); ``synth`` names the workloads and draws their seeded
synthetic inputs.  Importing this package does not load the CUDA library;
``runtime.load()`` does, and fails loudly when it is missing.
"""
__all__ = ["runtime", "synth"]
