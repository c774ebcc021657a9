"""GB300-native KV-cache flush codecs (TurboQuantRVQ and KIVI) for sm_103a.

The compute path is the C-ABI CUDA library ``libvqflush.so`` built from
``csrc/``; :mod:`.api` is a thin ctypes binding with the same entry-point names.
"""
