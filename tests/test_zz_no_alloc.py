"""The allocation-free decode entry point (fattn_decode_paged_static).

Some callers cannot allocate device memory (plugins handed only their input and
output buffers, code inside a device-memory budget owned by someone else); for
them the library keeps the decode partials in a fixed 32 MiB device scratch.
This file is collected last so that, in a run stopping at the first failure,
every other test has already run. It must pass alone in a fresh process too.
"""
import ctypes

import pytest
import torch

from exact_tiled_attention_fattn_gb300 import inputs
from oracle import attention as orc
from tests.gpu_util import as_np, check, need_gpu


def _dev(x):
    return [t.cuda() for t in (x.q, x.kcache, x.vcache, x.block_table, x.seqlens)]


@pytest.mark.gpu
def test_static_scratch_decode_matches_workspace_decode_twice():
    """Two calls in a row with different shapes: each output equals the workspace entry
    point's (same kernels) and the fp64 oracle's, within the bf16 tolerances."""
    fa = need_gpu()
    cases = [
        (inputs.decode_paged(61, 4, 16, 4, 128, 16, (100, 9000), 9216, spare_pages=4), 16),
        (inputs.decode_paged(62, 3, 8, 2, 64, 16, None, 4096, spare_pages=2, lengths=[1, 4096, 700]), 37),
    ]
    for x, S in cases:                                   # two calls in a row, different shapes
        q, kc, vc, bt, sl = _dev(x)
        o_ws, l_ws = fa.decode_paged(q, kc, vc, bt, sl, S, scale=x.scale)
        o, l = fa.decode_paged_static(q, kc, vc, bt, sl, S, scale=x.scale)
        assert fa.debug_read_status() == 0
        check(o, l, as_np(o_ws), as_np(l_ws), what=f"static scratch vs workspace S={S}")
        o_ref, l_ref = orc.decode_paged(x.q, x.kcache, x.vcache, x.block_table, x.seqlens, x.scale)
        check(o, l, o_ref, l_ref, what=f"static scratch vs oracle S={S}")


@pytest.mark.gpu
def test_static_scratch_rejects_problems_beyond_its_size():
    fa = need_gpu()
    x = inputs.decode_paged(63, 2, 8, 2, 128, 16, None, 256, spare_pages=1, lengths=[10, 200])
    q, kc, vc, bt, sl = _dev(x)
    S = 5000                                            # 2*8*5000*(128+1)*4 B > 32 MiB
    assert fa.decode_workspace_size(2, 8, 128, S) > fa.DECODE_STATIC_SCRATCH_BYTES
    with pytest.raises(fa.FattnError) as e:
        fa.decode_paged_static(q, kc, vc, bt, sl, S, scale=x.scale)
    assert e.value.status == fa.FATTN_ERR_WORKSPACE
    lib = fa.load_library()
    st = lib.fattn_decode_paged_static(None, None, None, None, None, 4, None, None, 2, 8, 2, 128, 16, 16, 1,
                                       0.1, ctypes.c_void_p(0))
    assert st == fa.FATTN_ERR_INVALID_ARG
