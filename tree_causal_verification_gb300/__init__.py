"""libjtree for GB300: one decode step of causal parallel tree drafting.

- ``jtree``: the Python binding of the C ABI (include/jtree.h).
- ``step``: the whole hot path (top-W -> expand -> mask -> attention ->
  accept) over preallocated device buffers.
- ``synth``: seeded synthetic inputs.
- ``build``: compiles libjtree.so for sm_103a.
"""
from . import synth  # noqa: F401

__all__ = ["jtree", "step", "synth", "build"]
