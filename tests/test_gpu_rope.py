"""GPU: the rotary prologue against the oracle, bit for bit.

The bf16 path hands the attention the nearest-even bf16 of the rotation with fp64 cos/sin
("Accelerating Video Generation Inference with Sequential-Parallel 3D Positional Encoding Using
a Global Time Index", section 2: the fused projection + RoPE step writes the rotated q and k as
the pipeline's bf16 tensors). The oracle rotates in fp64 and rounds once; the library's
rotated k (and q, when the tables are too large for the pair kernel's shared memory) is read
back from the step's workspace, where ditango_attn_step leaves it, and must match exactly.
The sizes cover every frame, row and column of the 720p-shaped latent (21 x 45 x 80) and of a
2 x 1000 latent whose tables send q through the pre-pass too; about one channel pair in a
thousand takes the kernel's exact slow path, so each case exercises it thousands of times.
"""
import numpy as np
import pytest
import torch

import attention_state_reuse_gb300 as dt
import oracle
from attention_state_reuse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dt.build()
    dt.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _rotated_from_workspace(w, q_in_prepass):
    dev = torch.device("cuda")
    B, N, H, d, P = w.B, w.N, w.H, w.d, w.P
    dtt, dhh, dww = w.rope_dims
    rope = dt.RopeTables(w.start_frame + w.T, w.Hl, w.Wl, dtt, dhh, dww,
                         start_frame=w.start_frame, device=dev)
    plan = dt.Plan(N, P)
    q_np, k_np, v_np = wl.InputStream(w).next()
    q, k, v = (torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in (q_np, k_np, v_np))
    cO, cL = dt.new_state_cache(B, H, P, N, d, torch.bfloat16, dev)
    out = torch.empty_like(q)
    nbytes = dt.workspace_size(plan, B, H, d, torch.bfloat16, True)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    dt.attn_step(plan, q, k, v, cO, cL, out, rope=rope, softmax_scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert dt.device_status() == (0, 0)
    one = (B * N * H * d * 2 + 255) // 256 * 256  # each rotated copy, 256-byte aligned
    k_rot = ws[: B * N * H * d * 2].view(torch.bfloat16).view(B, N, H, d)
    got = {"k": k_rot.float().cpu().numpy()}
    src = {"k": k_np}
    if q_in_prepass:
        q_rot = ws[one: one + B * N * H * d * 2].view(torch.bfloat16).view(B, N, H, d)
        got["q"] = q_rot.float().cpu().numpy()
        src["q"] = q_np
    return got, src


@pytest.mark.parametrize("name,kw,q_in_prepass", [
    ("long_720p", dict(H=3), False),                                   # 21 x 45 x 80, frames 0..20
    ("wan14b_layer", dict(H=2, T=1, Hl=2, Wl=1000, start_frame=7), True),  # wide tables
    ("wan14b_layer", dict(H=2, T=5, Hl=30, Wl=52, start_frame=16), False),  # frames 16..20
])
def test_rotated_inputs_match_oracle_bit_for_bit(name, kw, q_in_prepass):
    w = wl.scaled(wl.get(name), f"{name}_rope", steps=1, **kw)
    got, src = _rotated_from_workspace(w, q_in_prepass)
    dtt, dhh, dww = w.rope_dims
    for key, x in src.items():
        ref = oracle.rope_apply(x, w.Hl, w.Wl, w.start_frame, dtt, dhh, dww,
                                round_mode=oracle.ROUND_BF16)
        bad = np.argwhere(got[key] != ref)
        assert bad.size == 0, (key, len(bad), bad[:5].tolist())
