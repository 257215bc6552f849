"""pa_attention_noalloc: the attention step for callers that cannot allocate
device memory per step -- an engine that has given all free HBM to its
KV-cache pool, or code that must not call cudaMalloc / cudaFree mid-step
because they can synchronise the device.  It runs on the library's fixed
device scratch and must give what pa_attention gives with a workspace, on two
calls in a row (the calls share that scratch and it keeps the previous
call's contents).
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_82_gb300 as pa
import workloads
from tests._gpu_step import ATOL, gpu_step, owned_rows

pytestmark = pytest.mark.gpu

STEPS = {
    "decode": lambda: workloads.config2(batch=8, lo=17, hi=700,
                                       num_blocks=600),
    "mixed": lambda: workloads.config4(num_decodes=10, lo=100, hi=400,
                                      prefix=80, chunk=150, num_blocks=600),
    "fp8": lambda: workloads.config5(batch=4, lo=300, hi=2000,
                                    num_blocks=700),
}


@pytest.mark.parametrize("name", sorted(STEPS))
def test_noalloc_matches_attention_on_two_calls(name):
    wl = STEPS[name]()
    ref, kc, vc, md, flags = gpu_step(wl)   # copies, writes, pa_attention
    assert flags == 0
    dev = lambda x: torch.from_numpy(x).cuda()  # noqa: E731
    rows = owned_rows(md)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        pa.pa_attention_noalloc(
            wl.q.cuda(), kc, vc, dev(md["block_tables"]), dev(md["seq_lens"]),
            dev(md["query_start_loc"]), md["max_query_len"],
            md["max_seq_len"], wl.scale, wl.k_scale, wl.v_scale, out=out,
            cache_dtype=wl.cache_dtype)
        assert pa.pa_get_device_error() == 0
        a = out.float().cpu().numpy()[rows]
        b = ref.float().cpu().numpy()[rows]
        assert np.isfinite(a).all()
        assert float(np.abs(a - b).max()) <= ATOL[wl.cache_dtype]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = pa.load_library()
    f = lib.pa_attention_noalloc
    P, i64, i32, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                        ctypes.c_float)
    f.argtypes = [P, i32, P, P, i32, i64, i32, i32, i32, i32, P, i32, P, P,
                  i32, i64, i32, i32, f32, f32, f32, P, P]
    f.restype = i32
    need = pa.pa_attention_workspace_size(1 << 22, 32, 8, 128, 1 << 22, 1,
                                          4096)
    assert need > pa_scratch_bytes()
    kc = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
    small = torch.zeros(16, dtype=torch.int32, device="cuda")
    q = torch.zeros(2, 32, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    # far more sequences than the buffers hold: rejected on the host, before
    # anything reads them
    st = f(q.data_ptr(), pa.PA_BF16, kc.data_ptr(), kc.clone().data_ptr(),
           pa.PA_BF16, 4, 16, 32, 8, 128, small.data_ptr(), 256,
           small.data_ptr(), small.data_ptr(), 1 << 22, 1 << 22, 1, 4096,
           0.1, 1.0, 1.0, out.data_ptr(),
           torch.cuda.current_stream().cuda_stream)
    assert st == pa.PA_ERR_INVALID_ARG
    assert pa.pa_get_device_error() == 0


def pa_scratch_bytes():
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                       "pa.h")
    m = re.search(r"#define PA_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* "
                  r"(\d+)u\)", open(hdr).read())
    return int(m.group(1)) * int(m.group(2)) * int(m.group(3))
