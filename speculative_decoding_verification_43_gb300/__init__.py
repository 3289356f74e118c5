"""GB300-native batched speculative-decoding verifier.

The verifier step (accept/reject with residual or bonus draws, ragged compaction, and the
gamma controller) runs in hand-written sm_103a CUDA kernels behind the C ABI declared in
include/spec_verify.h. This package is the thin Python binding: ``api`` marshals torch tensors
into that ABI; ``workloads`` builds seeded synthetic inputs. Importing ``api`` loads
libspecverify.so and fails loudly if it has not been built.
"""
__all__ = ["api", "workloads", "build"]
