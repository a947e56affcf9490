"""forge_dgrad_noalloc: the input gradient dX = dY W with its split partials in
the library's static device scratch instead of a pool allocation.  It must
give forge_dgrad's result bit for bit at the same split count, fall back to
fewer splits when the scratch is too small, match the oracle, and leave the
device's free memory unchanged."""
import numpy as np
import pytest
import torch

from weight_gradient_gemm_gb300 import forge as F
from weight_gradient_gemm_gb300.inputs import bf16_bits, make_step_inputs

from .gpu_util import DEV, require_gpu
from .test_gpu_dgrad import check_dx

pytestmark = pytest.mark.gpu

SCRATCH = 32 << 20   # bytes of fp32 partials the library reserves per device


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(seed, bt, d_in, d_out):
    s = make_step_inputs(90 + seed, 0, 1, bt, d_in, d_out, dy_std=1e-3, with_w=True,
                         spike_frac=0.01)
    return s.dy.to(DEV), s.w.to(DEV), s


def _both(dy, w, bt, d_in):
    a = torch.full((bt, d_in), float("nan"), dtype=torch.bfloat16, device=DEV)
    b = torch.full_like(a, float("nan"))
    F.dgrad(dy, w, a)
    F.dgrad_noalloc(dy, w, b)
    assert F.device_error() == 0
    return a, b


@pytest.mark.parametrize("splits", [None, "2", "3", "4"])
@pytest.mark.parametrize("bt,d_in,d_out", [(200, 264, 4104), (512, 4096, 4096), (77, 136, 2048)])
def test_noalloc_equals_dgrad(bt, d_in, d_out, splits, tune):
    # every case here fits the scratch, so both use the same split count
    if splits is not None:
        tune(splits=int(splits))
    dy, w, s = _inputs(1, bt, d_in, d_out)
    a, b = _both(dy, w, bt, d_in)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    check_dx(bf16_bits(b.cpu()), bf16_bits(s.dy), bf16_bits(s.w), label=f"noalloc S={splits}")


def test_noalloc_uses_fewer_splits_when_the_scratch_is_too_small(tune):
    # Llama-3.1-8B gate projection at 512 tokens with 8 splits wants
    # 32 pair tiles x 2 CTAs x 8 x 128 KB = 64 MiB of partials: the variant
    # runs with 4 (32 MiB) and then equals forge_dgrad with 4 splits
    bt, d_out, d_in = 512, 14336, 4096
    assert 32 * 2 * 8 * 128 * 256 * 4 > SCRATCH >= 32 * 2 * 4 * 128 * 256 * 4
    dy, w, s = _inputs(2, bt, d_in, d_out)
    tune(splits=8)
    b = torch.full((bt, d_in), float("nan"), dtype=torch.bfloat16, device=DEV)
    F.dgrad_noalloc(dy, w, b)
    tune(splits=4)
    a = torch.full_like(b, float("nan"))
    F.dgrad(dy, w, a)
    assert F.device_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    rows = np.array([0, 1, 127, 128, 255, 256, 383, 511])
    check_dx(bf16_bits(b.cpu())[rows], bf16_bits(s.dy), bf16_bits(s.w), rows,
             label="noalloc gate")


def test_noalloc_runs_unsplit_when_not_even_two_splits_fit(tune):
    # Llama-3.1-8B down projection's dX at 512 tokens (d_in = 14336): 112 pair
    # tiles x 2 CTAs x 2 splits x 128 KB = 56 MiB of partials, more than the
    # scratch holds, so the variant runs unsplit and equals forge_dgrad with
    # one split
    bt, d_out, d_in = 512, 4096, 14336
    assert 112 * 2 * 2 * 128 * 256 * 4 > SCRATCH
    dy, w, s = _inputs(6, bt, d_in, d_out)
    tune(splits=2)
    b = torch.full((bt, d_in), float("nan"), dtype=torch.bfloat16, device=DEV)
    F.dgrad_noalloc(dy, w, b)
    tune(splits=1)
    a = torch.full_like(b, float("nan"))
    F.dgrad(dy, w, a)
    assert F.device_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    rows = np.array([0, 1, 127, 128, 255, 256, 383, 511])
    check_dx(bf16_bits(b.cpu())[rows], bf16_bits(s.dy), bf16_bits(s.w), rows,
             label="noalloc down unsplit")


def test_noalloc_leaves_free_memory_unchanged(tune):
    tune(splits=4)
    cases = [_inputs(3 + i, bt, d_in, d_out) + ((bt, d_in),)
             for i, (bt, d_in, d_out) in enumerate([(512, 4096, 14336), (256, 1024, 4096)])]
    outs = [torch.empty(shape, dtype=torch.bfloat16, device=DEV) for *_, shape in cases]
    for (dy, w, _, _), o in zip(cases, outs):   # first calls load the module's kernels
        F.dgrad_noalloc(dy, w, o)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for (dy, w, _, _), o in zip(cases, outs):
            F.dgrad_noalloc(dy, w, o)
    torch.cuda.synchronize()
    assert F.device_error() == 0
    assert torch.cuda.mem_get_info()[0] == free0
