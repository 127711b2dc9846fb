"""GB300-native paged KV-cache decode path (sm_103a).

The compute lives in ``libpagedkv.so`` (C ABI declared in ``include/pagedkv.h``);
``binding`` is its ctypes front end with the same names.  Importing this
package loads nothing; the first binding call loads the library and raises if
it has not been built.
"""

__all__ = ["binding"]
