"""GPU parity of moe_combine_add_rmsnorm (combine fused with the next layer's
residual add and RMSNorm) against the oracle: the oracle's layer sum, then its
add + RMSNorm in fp64; both outputs within 1e-2 relative Frobenius norm, pad
rows +0.0; and the fused residual output agrees with the unfused combine
output plus the residual to bf16 rounding."""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import MEDIUM, TOL, bf16_bits_to_f64, bf16_to_np, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("shape,R,pads", [(synth.TINY, 8, ()), (MEDIUM, 37, (0, 36))])
def test_add_rmsnorm_matches_oracle(shape, R, pads):
    wl = synth.Workload("an", shape, rows=R, pads=tuple(pads))
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    h = synth.to_numpy(t_cpu)
    cfg = m.Config.from_shape(shape)
    dev = torch.device("cuda")
    K, H, E = shape.topk, shape.hidden, shape.n_experts
    ids = torch.empty((R, K), dtype=torch.int32, device=dev)
    w = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.empty((R, E), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids, w, logits)
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids, ub)
    ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    ys = torch.empty((R * K, H), dtype=torch.float32, device=dev)
    ysh = torch.empty((R, H), dtype=torch.float32, device=dev)
    m.moe_expert_ffn_fp8(cfg, t["x"], m.Weights.from_tensors(t), ub, ys, ysh, ws)
    rng = np.random.default_rng(60)
    residual = torch.from_numpy(rng.normal(0, 1, (R, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    gamma = torch.from_numpy(rng.uniform(0.5, 1.5, H).astype(np.float32)).cuda()
    ro = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=dev)
    no = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=dev)
    m.moe_combine_add_rmsnorm(cfg, ys, ysh, w, ub, residual, gamma, 1e-5, ro, no)
    out = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    m.moe_combine(cfg, ys, ysh, w, ub, out)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    ref = oracle.moe_layer(shape, h)
    valid = h["row_valid"] != 0
    res_bits = bf16_to_np(residual.cpu())
    ro_ref, no_ref = oracle.add_rmsnorm(ref["y_acc"], res_bits, gamma.cpu().numpy(), 1e-5,
                                        h["row_valid"])
    got_ro, got_no = bf16_to_np(ro), bf16_to_np(no)
    assert rel_fro(bf16_bits_to_f64(got_ro)[valid], bf16_bits_to_f64(ro_ref)[valid]) <= TOL
    assert rel_fro(bf16_bits_to_f64(got_no)[valid], bf16_bits_to_f64(no_ref)[valid]) <= TOL
    assert np.all(got_ro[~valid] == 0) and np.all(got_no[~valid] == 0)
    # the fused residual output vs the unfused combine output plus the residual
    unfused = bf16_bits_to_f64(bf16_to_np(out)) + bf16_bits_to_f64(res_bits)
    assert rel_fro(bf16_bits_to_f64(got_ro)[valid], unfused[valid]) <= 2.0 ** -7
