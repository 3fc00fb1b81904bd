"""GB300-native context-parallel token layout and owner-gradient return.

The compute path is the C ABI in ``include/cpt.h`` (libcpt.so, hand-written
CUDA for sm_103a); ``context_attention_token_gb300.cpt`` is its Python
binding. ``synth`` holds the seeded synthetic input generators and ``build``
compiles the library in-tree.

Attribute access on the package (``context_attention_token_gb300.cpt_grad_return``
and friends) loads the binding lazily; it raises ImportError when the library
has not been built.
"""

__all__ = ["cpt", "synth", "build"]


def __getattr__(name):
    if name.startswith("cpt_") or name.startswith("CPT_") or name in ("Plan", "Epoch", "CptError"):
        from . import cpt as _cpt

        return getattr(_cpt, name)
    raise AttributeError(name)
