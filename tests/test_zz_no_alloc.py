"""pa_attention_noalloc: the attention step for callers that cannot allocate
device memory per step -- an engine that has given all free HBM to its
KV-cache pool, or code that must not call cudaMalloc / cudaFree mid-step
because they can synchronise the device.  It runs on the library's fixed
device scratch and must give what pa_attention gives with a workspace, on two
calls in a row (the calls share that scratch and it keeps the previous
call's contents).
"""
import ctypes

import pytest
import torch

import paged_kv_cache_82_gb300 as pa
import workloads
import oracle
from tests._gpu_step import assert_close, gpu_step, owned_rows

STEPS = {
    # one request: the workspace is then the fixed floor of split-K partial
    # slots that every decode step needs, whatever its batch
    "decode_batch1": lambda: workloads.config2(batch=1, lo=3000, hi=3000,
                                              num_blocks=300),
    "decode": lambda: workloads.config2(batch=8, lo=17, hi=700,
                                       num_blocks=600),
    "mixed": lambda: workloads.config4(num_decodes=10, lo=100, hi=400,
                                      prefix=80, chunk=150, num_blocks=600),
    "fp8": lambda: workloads.config5(batch=4, lo=300, hi=2000,
                                    num_blocks=700),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(STEPS))
def test_noalloc_matches_attention_on_two_calls(name):
    wl = STEPS[name]()
    ref, kc, vc, md, flags = gpu_step(wl)   # copies, writes, pa_attention
    assert flags == 0
    oracle_out, *_ = oracle.run_step(wl)
    dev = lambda x: torch.from_numpy(x).cuda()  # noqa: E731
    rows = torch.from_numpy(owned_rows(md)).cuda()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        pa.pa_attention_noalloc(
            wl.q.cuda(), kc, vc, dev(md["block_tables"]), dev(md["seq_lens"]),
            dev(md["query_start_loc"]), md["max_query_len"],
            md["max_seq_len"], wl.scale, wl.k_scale, wl.v_scale, out=out,
            cache_dtype=wl.cache_dtype)
        assert pa.pa_get_device_error() == 0
        # the same kernels on the same inputs: the same bits as pa_attention
        # (results are deterministic), so stale scratch cannot hide
        assert torch.equal(out[rows].view(torch.int16),
                           ref[rows].view(torch.int16))
        # and within the bar of the fp64 oracle
        assert_close(out, oracle_out, md, wl.cache_dtype, wl.q_dtype)


@pytest.mark.gpu
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


def _cpu_step():
    i32 = dict(dtype=torch.int32)
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16)
    return dict(q=q, k_cache=kc, v_cache=kc.clone(),
                block_tables=torch.zeros(2, 4, **i32),
                seq_lens=torch.ones(2, **i32),
                query_start_loc=torch.tensor([0, 1, 2], **i32),
                max_query_len=1, max_seq_len=1, scale=0.1,
                out=torch.empty_like(q))


@pytest.mark.parametrize("bad", ["strided_q", "int64_seq_lens", "short_qsl",
                                 "out_dtype"])
@pytest.mark.parametrize("fn", ["pa_attention", "pa_attention_noalloc"])
def test_binding_refuses_tensors_the_abi_would_misread(fn, bad):
    # both wrappers check layouts and metadata types before any pointer is
    # taken (no GPU needed: the check comes first)
    a = _cpu_step()
    if bad == "strided_q":
        a["q"] = torch.zeros(2, 16, 128, dtype=torch.bfloat16)[:, ::2]
    elif bad == "int64_seq_lens":
        a["seq_lens"] = a["seq_lens"].long()
    elif bad == "short_qsl":
        a["query_start_loc"] = a["query_start_loc"][:2]
    else:
        a["out"] = a["out"].float()
    with pytest.raises(ValueError):
        getattr(pa, fn)(**a)
