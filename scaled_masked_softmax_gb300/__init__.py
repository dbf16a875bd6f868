"""GB300 (sm_103a) fused ScaledMaskSoftmax: CUDA kernels behind a C ABI (libsms).

    from scaled_masked_softmax_gb300 import scaled_mask_softmax
    y = scaled_mask_softmax(scores, mask=None, scale=1/8, is_causal=True)
    y.backward(dy)
"""
from .binding import (  # noqa: F401
    PATH_NAMES, SMS_BF16, SMS_F16, SMS_F32, SMS_PATH_AUTO, SMS_PATH_CTA, SMS_PATH_ONLINE, SMS_PATH_RING, SMS_PATH_STREAM, SMS_PATH_WARP, SmsError,
    sms_attention_backward, sms_attention_backward_workspace, sms_attention_forward, sms_backward, sms_backward_lengths, sms_device_error, sms_forward, sms_forward_bool, sms_forward_lengths, sms_last_error, sms_last_path, sms_launch_count, sms_set_test_stall,
    sms_select_path, sms_set_forced_path, sms_set_grid_limit, sms_status_string, sms_version)
from .functional import ScaledMaskSoftmaxFunction, backward, forward, mask_layout, scaled_mask_softmax  # noqa: F401
from .attention import FusedAttentionFunction, attention_backward, attention_forward, fused_attention  # noqa: F401,E402
