"""GB300 (sm_103a) LRKV factored-cache attention.

The compute path lives in the CUDA shared library built from `csrc/`; the
Python side (`lrkv`) only marshals arguments into its C ABI.  Importing this
package does not load the library; the first call into `lrkv` does, and it
raises if the library has not been built.
"""
__all__ = ["inputs", "lrkv"]
