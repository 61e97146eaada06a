"""Tree-verify gated-DeltaNet step for GB300 (sm_103a).

The compute lives in ``liblbx.so`` (C ABI, declared in ``include/lbx.h``);
``tree_verify_linear_gb300.lbx`` is its thin Python binding.  Importing the
package loads nothing: the library is loaded on first use, and a missing
library raises instead of falling back to anything else.
"""
