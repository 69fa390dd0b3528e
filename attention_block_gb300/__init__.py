"""GB300-native fused single-token decode attention block.

The compute path is the CUDA library ``libcf.so`` (sources in ``csrc/``, C ABI
in ``include/cf.h``); ``binding`` is its ctypes binding and ``synth`` draws
the seeded synthetic inputs.  Importing this package loads nothing; the
library is loaded (and built if stale) on first use, and any failure to load
it raises -- there is no fallback path.
"""
from . import binding  # noqa: F401
from .binding import (CF_BF16, CF_F16, CF_F32, CF_OK, CfError, DecodeAttnBlock,  # noqa: F401
                      cf_create, cf_decode_attn_block, cf_destroy, cf_get_launch_info,
                      cf_get_status, cf_set_debug, cf_strerror, make_config)
