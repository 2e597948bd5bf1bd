"""The allocation-free attention entry point against the regular one.

mla_decode_attend_noalloc exists for callers that cannot allocate device
memory (code inside another framework's allocator, or a runtime that forbids
cudaMalloc on its hot path): it runs the same decode and combine with the
split partials in the library's own device array.  Its output must match the
regular mla_decode_fwd + mla_combine path within the bf16 tolerance of the
other parity tests, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result).  The file name
makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_72_b300 import build
    build.build()


def _rel(got, ref):
    got = got.float().cpu().numpy()
    ref = ref.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def test_noalloc_matches_regular_path_on_two_calls():
    from mla_latent_kv_72_b300 import binding as C
    from mla_latent_kv_72_b300.workload import DeviceWorkload

    cases = [mi.scaled(mi.workload(3), B=3, L=900),
             mi.scaled(mi.workload(4), B=5, L_range=(1, 700))]
    for w in cases:
        dw = DeviceWorkload(w, device="cuda")
        dw.absorb()
        dw.attend()
        dw.combine()
        torch.cuda.synchronize()
        ref_lat, ref_lse = dw.o_lat.clone(), dw.lse.clone()
        for _ in range(2):
            o_lat = torch.full_like(dw.o_lat, float("nan"))
            lse = torch.full_like(dw.lse, float("nan"))
            C.mla_decode_attend_noalloc(dw.q_cat, dw.kv, dw.block_table, dw.seq_lens,
                                        dw.num_parts, o_lat, lse, dev_status=dw.status)
            torch.cuda.synchronize()
            assert dw.check_status() == 0
            assert _rel(o_lat, ref_lat) <= TOL
            assert _rel(lse, ref_lse) <= TOL


def test_noalloc_rejects_sizes_beyond_its_array():
    from mla_latent_kv_72_b300 import binding as C
    from mla_latent_kv_72_b300.workload import DeviceWorkload

    w = mi.scaled(mi.workload(3), B=2, L=64)
    dw = DeviceWorkload(w, device="cuda")
    big_b = 300   # (300 + parts - 1) * 128 * 512 floats > 16 Mi
    L = C.lib()
    st = L.mla_decode_attend_noalloc(
        dw.q_cat.data_ptr(), C.MLA_BF16, C.ctypes.byref(dw.kv), dw.block_table.data_ptr(),
        dw.block_table.shape[1], dw.seq_lens.data_ptr(), big_b, w.h, dw.num_parts, 0.0,
        dw.o_lat.data_ptr(), C.MLA_BF16, None, None, None)
    assert st == -4   # MLA_ERR_SHAPE, nothing launched
