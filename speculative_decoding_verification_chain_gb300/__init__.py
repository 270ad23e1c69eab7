"""GB300-native speculative-decoding verify-and-accept.

The CUDA library (``libspecverify.so``, C ABI declared in ``include/spec_verify.h``)
does every step of the path; this package only marshals arguments to it.
"""
