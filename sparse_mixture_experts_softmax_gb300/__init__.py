"""GB300-native (sm_103a) sparse top-k mixture-of-experts training step.

The layer lives in the CUDA library ``libmoe_gb300.so`` behind the C ABI of
``include/moe.h``; ``binding`` is its thin ctypes binding and ``layer`` a small
helper that owns the device buffers of one layer.
"""

from .binding import (MoEError, make_config, make_grads, make_params, make_weights,  # noqa: F401
                      moe_backward, moe_device_status, moe_dispatch_noalloc, moe_forward,
                      moe_get_hidden, moe_get_intermediates, moe_get_routing, moe_grouped_gemm,
                      moe_host_staging_size, moe_last_launch_count, moe_status_string,
                      moe_train_step, moe_train_step_host, moe_train_steps_host,
                      moe_workspace_size)
