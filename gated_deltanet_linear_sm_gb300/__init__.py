"""GB300-native Gated DeltaNet speculative / MTP decode step.

The compute is the sm_103a CUDA kernel in libgdnspec (C ABI, include/gdnspec.h);
this package holds its Python binding, its build step and the seeded
synthetic-input generator.
"""
from .binding import (BF16, F16, F32, GdnError, LibraryMissing, gdn_dims, gdn_prefill,  # noqa: F401
                      gdn_prefill_chunked, gdn_spec_decode, gdn_spec_decode_conv, library_path, load_library, prepare, status_str, version)
