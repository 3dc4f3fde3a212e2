"""GB300-native data-parallel hot path of ZeRO stages 1-3 (emulated ranks).

The work lives in the C-ABI library ``libzero.so`` (include/zero.h); this
package is its thin binding.  Build the library with ``build.build()``.
"""
from .binding import *  # noqa: F401,F403
from .binding import Plan, ZeroError, adam_hp, header_functions  # noqa: F401
