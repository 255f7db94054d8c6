"""GB300 (sm_103a) library for batched speculative-decoding verification.

The compute path is the C-ABI shared library libspecverify.so (CUDA kernels in
csrc/, declared in include/spec_verify.h); ``verify`` is its thin ctypes
binding. Importing the package does not load the library: the first call
does, and raises SpecVerifyError if it has not been built.
"""

from .verify import (  # noqa: F401
    RULE_EXACT, RULE_POWER, RULE_RELAXED,
    STATUS_BAD_PAGE, STATUS_BAD_PARENT, STATUS_BAD_TOKEN, STATUS_CAPPED, STATUS_DEPTH_EXCEEDED,
    STATUS_NONFINITE_ROW, STATUS_STOPPED, STATUS_TIMEOUT, STATUS_ZERO_MASS, SV_ERR_TIMEOUT,
    SpecVerifyError, library_path, load_library,
    spec_kv_compact, spec_tree_build, spec_verify_check_status, spec_verify_greedy, spec_verify_greedy_early,
    spec_verify_greedy_host,
    spec_verify_sample, spec_verify_selftest_wait, spec_verify_tree, spec_verify_workspace_size,
)
