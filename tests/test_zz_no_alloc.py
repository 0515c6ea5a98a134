"""oscar_decode_static_workspace: decode for callers that cannot allocate device memory.

Some callers can't hand the decode a workspace. An engine may pass only the
step's inputs and outputs. A serving loop may own all device memory in its own
allocator. A step may run under CUDA stream capture, where cudaMalloc is not
allowed. For them the library keeps its scratch in one static device array.
These tests call that entry point through the C ABI. They check its output
against oscar_decode's (same kernels, caller workspace) on two calls in a row
with different inputs, so contents left by the first call can't leak into the
second. They also check that sizes beyond the array are rejected. This file
is named to be collected last.
"""

import numpy as np
import pytest
import torch

import cases
from bit_kv_cache_write_gb300 import oscar as O

pytestmark = pytest.mark.gpu


def _tensors(case, dev):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(case.q).to(torch.bfloat16), int2_pool=t(case.int2_pool), int2_tables=t(case.int2_tables),
                hist_len=t(case.hist_lens), bf16_pool=t(case.bf16_pool).to(torch.bfloat16),
                bf16_tables=t(case.bf16_tables), bf16_len=t(case.bf16_lens))


def test_static_workspace_matches_caller_workspace_on_two_calls_in_a_row(cuda):
    cfg = cases.workload("qwen3_8b_bs1_100k")
    first = cases.DecodeCase(cfg, [3001], [320])
    second = cases.DecodeCase(cfg, [700, 1900], [320, 200], layer=1)
    ctx = O.Oscar(n_layers=2, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"])
    for layer, case in ((0, first), (1, second)):
        ctx.calibrate_upload(layer, case.rk, case.rv, case.tk, case.tv)

    for layer, case in ((0, first), (1, second)):
        a = _tensors(case, cuda)
        B, mh = len(case.hist_lens), int(case.hist_lens.max())
        ws = torch.empty(ctx.decode_workspace_size(B, mh), dtype=torch.uint8, device=cuda)
        want = torch.empty(B, cfg["h_q"], cfg["d"], dtype=torch.float32, device=cuda)
        got = torch.full_like(want, float("nan"))
        ctx.decode(layer, a["q"], a["int2_pool"], a["int2_tables"], a["hist_len"], mh, a["bf16_pool"],
                   a["bf16_tables"], a["bf16_len"], want, ws)
        ctx.decode_static_workspace(layer, a["q"], a["int2_pool"], a["int2_tables"], a["hist_len"], mh,
                                    a["bf16_pool"], a["bf16_tables"], a["bf16_len"], got)
        torch.cuda.synchronize()
        cases.check_decode(got.cpu().numpy(), want.cpu().numpy())


def test_static_workspace_rejects_sizes_beyond_its_maximum(cuda):
    cfg = cases.workload("tiny")
    li, (rk, rv, tk, tv) = cases.calibration(cfg)
    ctx = O.Oscar(n_layers=1, n_q_heads=cfg["h_q"], n_kv_heads=cfg["h_kv"], head_dim=cfg["d"], group=cfg["group"])
    ctx.calibrate_upload(0, rk, rv, tk, tv)
    batch = 4096
    assert ctx.decode_workspace_size(batch, 1024) > 8 << 20
    z = lambda *s, dt=torch.int32: torch.zeros(*s, dtype=dt, device=cuda)
    with pytest.raises(O.OscarError) as e:
        ctx.decode_static_workspace(0, z(batch, 4, 64, dt=torch.bfloat16), z(4096, dt=torch.uint8), z(batch, 64),
                                    z(batch), 1024, z(2 * 2 * 2 * 16 * 64, dt=torch.bfloat16), z(batch, 20), z(batch),
                                    z(batch, 4, 64, dt=torch.float32))
    assert e.value.status == -7
    assert "static workspace" in str(e.value)
