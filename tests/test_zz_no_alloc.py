"""The workspace-free decode entry point, for callers that cannot allocate device memory in
their decode step (a loop that must not call cudaMalloc, a process whose memory belongs to
another allocator, an embedding that only lends its input and output buffers).

It must give the same answer as attn_decode_splitkv with a caller workspace, call after call:
the library's fixed scratch keeps the previous call's partial states, and a second call with
different sequences must not see them.  This file is collected last on purpose."""
import numpy as np
import pytest

import synthetic as syn
from parity import check_rows

pytestmark = pytest.mark.gpu


def _decode_pair(attn, lengths, Hq, Hkv, d, dt, seed, split=512):
    import torch

    cfg = syn.DecodeConfig("noalloc", len(lengths), Hq, Hkv, d, dt, seed,
                           lengths_override=tuple(lengths))
    q, kc, vc = cfg.host_inputs()
    cu = torch.from_numpy(syn.cu_seqlens(lengths)).cuda()
    qt, kt, vt = (syn.bits_to_tensor(x, dt, "cuda") for x in (q, kc, vc))
    ref_o, ref_l = attn.attn_decode_splitkv(qt, kt, vt, cu, max(lengths), split_size=split,
                                            scale=cfg.scale)
    o = torch.full_like(qt, float("nan"))
    lse = torch.full((len(lengths), Hq), float("nan"), device="cuda")
    o, lse = attn.attn_decode_splitkv_static(qt, kt, vt, cu, max(lengths), o=o, lse=lse,
                                             split_size=split, scale=cfg.scale)
    assert attn.attn_poll_status() == 0
    return [x.float().cpu().numpy().astype(np.float64) for x in (o, lse, ref_o, ref_l)]


def test_static_scratch_decode_matches_workspace_decode_twice():
    import exact_io_aware_09_gb300 as attn

    assert attn.attn_decode_static_scratch_bytes() == 32 << 20
    # first call: longer sequences; second call: different lengths, heads and type, so stale
    # partial states left in the shared scratch would show up
    for lengths, Hq, Hkv, d, dt, seed in (((3000, 1, 600, 4097), 16, 2, 128, "bf16", 61),
                                          ((513, 70, 2000), 8, 8, 64, "f16", 62)):
        o, lse, ref_o, ref_l = _decode_pair(attn, lengths, Hq, Hkv, d, dt, seed)
        check_rows(o.reshape(-1, d), lse.reshape(-1), ref_o.reshape(-1, d), ref_l.reshape(-1),
                   f"static-scratch decode {lengths}")


def test_static_scratch_call_allocates_no_device_memory():
    """Once the first call on the device has run, a call with preallocated o and lse takes no
    device memory: neither torch's allocator nor the driver's free-memory count moves."""
    import torch

    import exact_io_aware_09_gb300 as attn

    lengths, Hq, Hkv, d, dt = (700, 1900, 33), 16, 2, 128, "bf16"
    cfg = syn.DecodeConfig("noalloc", len(lengths), Hq, Hkv, d, dt, 63,
                           lengths_override=lengths)
    q, kc, vc = cfg.host_inputs()
    cu = torch.from_numpy(syn.cu_seqlens(lengths)).cuda()
    qt, kt, vt = (syn.bits_to_tensor(x, dt, "cuda") for x in (q, kc, vc))
    o = torch.empty_like(qt)
    lse = torch.empty((len(lengths), Hq), device="cuda", dtype=torch.float32)
    call = lambda: attn.attn_decode_splitkv_static(qt, kt, vt, cu, max(lengths), o=o, lse=lse,
                                                   scale=cfg.scale)
    call()
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    call()
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    assert attn.attn_poll_status() == 0
    assert after == before, (before, after)


def test_static_scratch_refuses_requests_that_do_not_fit():
    import torch

    import exact_io_aware_09_gb300 as attn

    q = torch.zeros((64, 64, 128), device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros((1024, 8, 128), device="cuda", dtype=torch.bfloat16)
    cu = torch.zeros(65, device="cuda", dtype=torch.int32)
    need = attn.attn_decode_workspace_bytes(64, 64, 32768, 512, 128)
    assert need > attn.attn_decode_static_scratch_bytes()
    with pytest.raises(attn.AttnError) as e:
        attn.attn_decode_splitkv_static(q, kc, kc, cu, 32768)
    assert e.value.status == -4
