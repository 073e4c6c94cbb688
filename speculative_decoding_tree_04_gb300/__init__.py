"""GB300-native tree-verify MLA-absorb attention (DDTree speculative decoding).

The compute lives in ``libtv.so`` (hand-written sm_103a CUDA behind a C ABI declared in
``include/tv.h``); ``speculative_decoding_tree_04_gb300.tv`` is the thin ctypes binding
with the same call names.  Importing this package loads nothing: the library is opened on
first use of the binding, which raises if it has not been built.
"""
__all__ = ["tv", "synth"]
