"""The Python binding without a GPU: every public op refuses host tensors (there is no CPU fallback:
the C ABI takes device pointers only), and the composite ops check dtypes and shapes before any
launch."""
import pytest
import torch

import mxfp8_precision_moe_gb300 as mx


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


OFFS = torch.tensor([64, 128], dtype=torch.int32)


@pytest.mark.parametrize("call", [
    lambda: mx.mxfp8_quantize_2d(bf(128, 64), mx.ROW | mx.COL, mx.SCALES_BLOCKED, OFFS),
    lambda: mx.mxfp8_quantize_3d_experts(bf(2, 64, 64)),
    lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), OFFS),
    lambda: mx.mxfp8_grouped_mm_dgrad(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), OFFS),
    lambda: mx.mxfp8_grouped_mm_wgrad(u8(64, 128), u8(4096), u8(64, 128), u8(4096), OFFS),
    lambda: mx.mxfp8_swiglu_bwd_quantize(bf(128, 64), bf(128, 64), bf(128, 64), OFFS),
    lambda: mx.to_mxfp8_then_scaled_grouped_mm(bf(128, 64), bf(2, 64, 64), OFFS),
    lambda: mx.mxfp8_swiglu_expert(bf(128, 64), bf(2, 64, 64), bf(2, 64, 64), bf(2, 64, 64), OFFS),
])
def test_host_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA"):
        call()


def test_composite_ops_check_dtypes_and_shapes_first():
    with pytest.raises(ValueError, match="bf16"):
        mx.to_mxfp8_then_scaled_grouped_mm(bf(128, 64).float(), bf(2, 64, 64), OFFS)
    with pytest.raises(ValueError, match="int32"):
        mx.to_mxfp8_then_scaled_grouped_mm(bf(128, 64), bf(2, 64, 64), OFFS.long())
    with pytest.raises(ValueError, match="bf16"):
        mx.mxfp8_swiglu_expert(bf(128, 64), bf(2, 64, 64).float(), bf(2, 64, 64), bf(2, 64, 64), OFFS)
    with pytest.raises(ValueError, match="shapes"):
        mx.mxfp8_swiglu_expert(bf(128, 64), bf(2, 64, 64), bf(2, 64, 64), bf(2, 32, 64), OFFS)
    with pytest.raises(ValueError, match="bf16"):
        mx.mxfp8_swiglu_bwd_quantize(bf(128, 64), bf(128, 64).float(), bf(128, 64), OFFS)


# shapes, offsets lengths and scale-buffer sizes are checked on the host before any call: the C ABI
# sees raw pointers only, so a short buffer would otherwise be read past its end on the device
@pytest.mark.parametrize("call,match", [
    (lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(4096), u8(2, 64, 32), u8(2, 2048), OFFS), "w_q"),
    (lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(4096), u8(3, 64, 64), u8(3, 2048), OFFS), "offs"),
    (lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(100), u8(2, 64, 64), u8(2, 2048), OFFS), "a_s"),
    (lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 100), OFFS), "w_s"),
    (lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), OFFS.long()), "offs"),
    (lambda: mx.mxfp8_grouped_mm_fwd(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), OFFS,
                                     out=bf(128, 32)), "out"),
    (lambda: mx.mxfp8_grouped_mm_fwd(bf(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), OFFS), "a_q"),
    (lambda: mx.mxfp8_grouped_mm_dgrad(u8(128, 64), u8(4096), u8(2, 64, 32), u8(2, 2048), OFFS), "wt_q"),
    (lambda: mx.mxfp8_grouped_mm_dgrad(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 10), OFFS), "wt_s"),
    (lambda: mx.mxfp8_grouped_mm_wgrad(u8(64, 128), u8(4096), u8(64, 96), u8(4096), OFFS), "aT_q"),
    (lambda: mx.mxfp8_grouped_mm_wgrad(u8(64, 128), u8(1000), u8(64, 128), u8(4096), OFFS), "doutT_s"),
    (lambda: mx.mxfp8_grouped_mm_wgrad(u8(64, 128), u8(4096), u8(64, 128), u8(4096), OFFS,
                                       dev_status=torch.zeros(1, dtype=torch.int64)), "dev_status"),
    (lambda: mx.mxfp8_grouped_mm_dgrad2(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), u8(128, 64), u8(100),
                                        u8(2, 64, 64), u8(2, 2048), OFFS), "dout2_s"),
    (lambda: mx.mxfp8_grouped_mm_swiglu_fwd(u8(128, 64), u8(4096), u8(2, 64, 64), u8(2, 2048), u8(2, 32, 64),
                                            u8(2, 2048), OFFS), "up weights"),
    (lambda: mx.mxfp8_quantize_2d(bf(128, 64), mx.ROW, mx.SCALES_BLOCKED, OFFS.reshape(2, 1)), "offs"),
    (lambda: mx.mxfp8_check_offsets(OFFS, 128, 32, None), "dev_status"),
    (lambda: mx.to_mxfp8_then_scaled_grouped_mm(bf(128, 64), bf(3, 64, 64), OFFS), "offs"),
    (lambda: mx.to_mxfp8_then_scaled_grouped_mm(bf(128, 64), bf(2, 64, 32), OFFS), "A \\[M, K\\]"),
    (lambda: mx.mxfp8_swiglu_expert(bf(128, 64), bf(3, 64, 64), bf(3, 64, 64), bf(3, 64, 64), OFFS), "offs"),
])
def test_shapes_and_buffer_sizes_are_checked_before_any_call(call, match):
    with pytest.raises(ValueError, match=match):
        call()
