"""The allocation-free attention entry point against the regular one.

Some callers cannot allocate device memory: code that runs inside another
framework's memory pool or allocator hooks, or a runtime that forbids
cudaMalloc on its hot path.  mla_decode_attend_noalloc serves them: it runs
the same decode and combine kernels as mla_decode_fwd + mla_combine, with the
split partials in the library's own fixed device array.  Same kernels on the
same inputs in the same order, so its outputs must equal the regular path's
bit for bit.  The calls alternate between two workloads with different
lengths, part layouts and slot counts (A, B, A), so each call follows one that
left different contents in the shared array: a stale slot would show.  The
file name makes pytest collect it last.
"""
import pytest
import torch

import mla_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_72_b300 import build
    build.build()


def _same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32),
                       b.contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32))


def test_noalloc_matches_regular_path_bit_for_bit():
    from mla_latent_kv_72_b300 import binding as C
    from mla_latent_kv_72_b300.workload import DeviceWorkload

    work = {
        "A": DeviceWorkload(mi.scaled(mi.workload(3), B=3, L=900), device="cuda", num_parts=5),
        "B": DeviceWorkload(mi.scaled(mi.workload(4), B=5, L_range=(1, 700)), device="cuda",
                            num_parts=11),
    }
    ref = {}
    for k, dw in work.items():
        dw.absorb()
        dw.attend()
        dw.combine()
        torch.cuda.synchronize()
        assert dw.check_status() == 0
        ref[k] = (dw.o_lat.clone(), dw.lse.clone())
    for k in ("A", "B", "A"):
        dw = work[k]
        o_lat = torch.full_like(dw.o_lat, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        C.mla_decode_attend_noalloc(dw.q_cat, dw.kv, dw.block_table, dw.seq_lens, dw.num_parts,
                                    o_lat, lse, dev_status=dw.status)
        torch.cuda.synchronize()
        assert dw.check_status() == 0
        assert _same_bits(o_lat, ref[k][0]), k
        assert _same_bits(lse, ref[k][1]), k


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
