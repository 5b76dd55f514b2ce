"""GPU router and dispatch vs the oracle: indices and permutations bit-exact."""

import numpy as np
import pytest
import torch

import synthetic
import quantized_routed_expert_03_gb300 as qre
from oracle import moe as omoe

from gpu_support import bits_to_bf16_tensor, check_routing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _route(H, E, k, T, seed, bias=None, layer=0):
    x_bits = synthetic.activations_bits(T, H, seed=seed, layer=layer)
    wr = synthetic.router_weights(E, H, seed=seed, layer=layer)
    shape = qre.make_shape(H, 128, E, k, 32)
    ws = torch.empty(max(qre.qre_workspace_size(shape, T), 256), dtype=torch.uint8, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    b = None if bias is None else torch.from_numpy(bias).to(DEV)
    qre.qre_route(shape, T, bits_to_bf16_tensor(x_bits, DEV), torch.from_numpy(wr).to(DEV), b, idx, w, ws)
    torch.cuda.synchronize()
    ref = omoe.route(omoe.bf16_bits_to_f64(x_bits), wr, bias, k)
    return idx.cpu().numpy(), w.cpu().numpy(), ref


@pytest.mark.parametrize("H,E,k,T", [(256, 16, 4, 4), (4096, 288, 8, 1), (4096, 288, 8, 8), (512, 64, 6, 13),
                                     (1024, 288, 8, 16), (4096, 288, 8, 300), (768, 1024, 16, 40)])
def test_route_matches_oracle(H, E, k, T):
    idx, w, ref = _route(H, E, k, T, seed=3)
    near = check_routing(idx, w, ref)
    assert near <= max(1, T // 500)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-6)


def test_route_zipf_bias_matches_oracle():
    H, E, k, T = 4096, 288, 8, 64
    bias = synthetic.zipf_bias(E, seed=0, layer=2)
    idx, w, ref = _route(H, E, k, T, seed=0, bias=bias, layer=2)
    check_routing(idx, w, ref)


@pytest.mark.slow
def test_route_prefill_8192_matches_oracle():
    idx, w, ref = _route(4096, 288, 8, 8192, seed=0)
    near = check_routing(idx, w, ref)
    assert near < 40


def test_route_exact_ties_go_to_lower_id():
    H, E, k, T = 256, 16, 4, 3
    x_bits = synthetic.activations_bits(T, H, seed=1)
    wr = np.tile(np.linspace(-0.1, 0.1, H, dtype=np.float32), (E, 1))
    shape = qre.make_shape(H, 128, E, k, 32)
    ws = torch.empty(max(qre.qre_workspace_size(shape, T), 256), dtype=torch.uint8, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    qre.qre_route(shape, T, bits_to_bf16_tensor(x_bits, DEV), torch.from_numpy(wr).to(DEV), None, idx, w, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), np.tile(np.arange(k), (T, 1)))
    np.testing.assert_allclose(w.cpu().numpy(), 0.25, rtol=0, atol=1e-7)


def _dispatch(idx_np, E, k):
    T = idx_np.shape[0]
    shape = qre.make_shape(256, 128, E, k, 32)
    P = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    out = {n: torch.full((m,), -7, **i32) for n, m in
           (("counts", E), ("offsets", E + 1), ("perm", P), ("inv_perm", P), ("active", E), ("n_active", 4))}
    ws = torch.empty(max(qre.qre_workspace_size(shape, T), 256), dtype=torch.uint8, device=DEV)
    qre.qre_dispatch(shape, T, torch.from_numpy(idx_np.astype(np.int32)).to(DEV), out["counts"], out["offsets"],
                     out["perm"], out["inv_perm"], out["active"], out["n_active"], ws)
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in out.items()}


@pytest.mark.parametrize("T,E,k", [(1, 288, 8), (4, 16, 4), (8, 288, 8), (128, 288, 8), (129, 288, 8),
                                   (1000, 64, 2), (8192, 288, 8), (4096, 1024, 16), (3, 5, 5)])
def test_dispatch_matches_oracle(T, E, k):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.sort(np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]), axis=1)
    got = _dispatch(idx, E, k)
    ref = omoe.dispatch(idx, E)
    n = ref["n_active"]
    for name in ("counts", "offsets", "perm", "inv_perm"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    assert got["n_active"][0] == n
    np.testing.assert_array_equal(got["active"][:n], ref["active"])


def test_dispatch_skewed_all_tokens_one_expert_set():
    T, E, k = 2000, 288, 8
    idx = np.tile(np.arange(100, 108), (T, 1))
    got = _dispatch(idx, E, k)
    ref = omoe.dispatch(idx, E)
    for name in ("counts", "offsets", "perm", "inv_perm"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    assert got["n_active"][0] == 8


def test_dispatch_bad_index_sets_status_without_fault():
    qre.qre_clear_device_status()
    idx = np.array([[0, 3], [1, 99]], dtype=np.int32)   # 99 >= E
    got = _dispatch(idx, 16, 2)
    st = qre.qre_read_device_status()
    qre.qre_clear_device_status()
    assert st & qre.QRE_DEV_BAD_INDEX
    assert got["counts"].sum() == 3


def test_empty_call_is_a_no_op():
    shape = qre.make_shape(256, 128, 16, 4, 32)
    qre.qre_route(shape, 0, None, None, None, None, None, None, 0)
    qre.qre_dispatch(shape, 0, None, None, None, None, None, None, None, None, 0)
    qre.qre_expert_ffn(shape, 0, None, None, None, None, None, None, None, None, 0)
    qre.qre_combine(shape, 0, None, None, None, None, None)


@pytest.mark.parametrize("H,E,k,T,bias", [(4096, 288, 8, 1, False), (4096, 288, 8, 8, True), (256, 16, 4, 4, False),
                                          (512, 64, 6, 7, True), (768, 1024, 16, 8, False), (512, 64, 6, 40, False),
                                          (4096, 288, 8, 1, True), (256, 5, 5, 1, False), (256, 37, 16, 1, True),
                                          (768, 1024, 16, 1, True), (512, 1000, 3, 1, False)])
def test_route_dispatch_equals_route_then_dispatch(H, E, k, T, bias):
    """qre_route_dispatch (selection and dispatch in one CTA for T <= 8, the two
    calls' kernels above) writes the same bits as qre_route then qre_dispatch."""
    shape = qre.make_shape(H, 128, E, k, 32)
    x = bits_to_bf16_tensor(synthetic.activations_bits(T, H, seed=6, layer=1), DEV)
    wr = torch.from_numpy(synthetic.router_weights(E, H, seed=6, layer=1)).to(DEV)
    b = torch.from_numpy(synthetic.zipf_bias(E, seed=6, layer=1, beta=0.05)).to(DEV) if bias else None
    ws = torch.empty(max(qre.qre_workspace_size(shape, T), 256), dtype=torch.uint8, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)

    def outs():
        return {"idx": torch.full((T, k), -1, **i32), "w": torch.full((T, k), -1.0, device=DEV),
                "counts": torch.full((E,), -1, **i32), "offsets": torch.full((E + 1,), -1, **i32),
                "perm": torch.full((T * k,), -1, **i32), "inv_perm": torch.full((T * k,), -1, **i32),
                "active": torch.full((E,), -1, **i32), "n_active": torch.full((4,), -1, **i32)}
    a, f = outs(), outs()
    qre.qre_route(shape, T, x, wr, b, a["idx"], a["w"], ws)
    qre.qre_dispatch(shape, T, a["idx"], a["counts"], a["offsets"], a["perm"], a["inv_perm"], a["active"],
                     a["n_active"], ws)
    qre.qre_route_dispatch(shape, T, x, wr, b, f["idx"], f["w"], f["counts"], f["offsets"], f["perm"], f["inv_perm"],
                           f["active"], f["n_active"], ws)
    torch.cuda.synchronize()
    n = int(a["n_active"][0].item())
    assert int(f["n_active"][0].item()) == n
    for name in ("idx", "w", "counts", "offsets", "perm", "inv_perm"):
        np.testing.assert_array_equal(f[name].cpu().numpy(), a[name].cpu().numpy(), err_msg=name)
    np.testing.assert_array_equal(f["active"][:n].cpu().numpy(), a["active"][:n].cpu().numpy())
    assert qre.qre_read_device_status() == 0


@pytest.mark.parametrize("E,k", [(16, 4), (288, 8), (1024, 16)])
def test_route_dispatch_one_token_exact_ties(E, k):
    """One token whose experts all score the same: the one-CTA selection and
    dispatch picks experts 0..k-1 (ties to the lower id), each with weight 1/k,
    and dispatches them in place (perm and inv_perm the identity)."""
    H = 256
    shape = qre.make_shape(H, 128, E, k, 32)
    x = bits_to_bf16_tensor(synthetic.activations_bits(1, H, seed=1), DEV)
    wr = torch.from_numpy(np.tile(np.linspace(-0.1, 0.1, H, dtype=np.float32), (E, 1))).to(DEV)
    ws = torch.empty(max(qre.qre_workspace_size(shape, 1), 256), dtype=torch.uint8, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    o = {"idx": torch.full((1, k), -1, **i32), "w": torch.full((1, k), -1.0, device=DEV),
         "counts": torch.full((E,), -1, **i32), "offsets": torch.full((E + 1,), -1, **i32),
         "perm": torch.full((k,), -1, **i32), "inv_perm": torch.full((k,), -1, **i32),
         "active": torch.full((E,), -1, **i32), "n_active": torch.full((4,), -1, **i32)}
    qre.qre_route_dispatch(shape, 1, x, wr, None, o["idx"], o["w"], o["counts"], o["offsets"], o["perm"],
                           o["inv_perm"], o["active"], o["n_active"], ws)
    torch.cuda.synchronize()
    g = {n: t.cpu().numpy() for n, t in o.items()}
    np.testing.assert_array_equal(g["idx"][0], np.arange(k))
    np.testing.assert_allclose(g["w"][0], 1.0 / k, rtol=1e-6, atol=0)
    np.testing.assert_array_equal(g["counts"], (np.arange(E) < k).astype(np.int32))
    np.testing.assert_array_equal(g["offsets"], np.minimum(np.arange(E + 1), k))
    np.testing.assert_array_equal(g["perm"], np.arange(k))
    np.testing.assert_array_equal(g["inv_perm"], np.arange(k))
    np.testing.assert_array_equal(g["active"][:k], np.arange(k))
    assert g["n_active"][0] == k


def _route_with_logits(H, E, k, T, x_bits, wr):
    """qre_route, plus the logits it leaves at the start of its workspace (the
    router writes them there before the selection reads them)."""
    shape = qre.make_shape(H, 128, E, k, 32)
    ws = torch.zeros(max(qre.qre_workspace_size(shape, T), 256), dtype=torch.uint8, device=DEV)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    qre.qre_route(shape, T, bits_to_bf16_tensor(x_bits, DEV), torch.from_numpy(wr).to(DEV), None, idx, w, ws)
    torch.cuda.synchronize()
    logits = ws[:T * E * 4].view(torch.float32).reshape(T, E).cpu().numpy()
    return idx.cpu().numpy(), w.cpu().numpy(), logits


@pytest.mark.parametrize("H,E,T", [(4096, 288, 1024), (256, 16, 2048), (768, 1000, 1100), (512, 300, 1030)])
def test_route_tensor_core_split_is_exact(H, E, T):
    """Long batches take the tensor-core logits (the fp32 router weights as three
    bf16 parts): with one-hot tokens every logit is a single weight, which the
    three exact part products must give back bit for bit."""
    rng = np.random.default_rng(E + T)
    wr = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    cols = (np.arange(T) * 37) % H
    x = np.zeros((T, H), np.float64)
    x[np.arange(T), cols] = 1.0
    x_bits = omoe.f32_to_bf16_bits(x.astype(np.float32))
    _, _, logits = _route_with_logits(H, E, 4, T, x_bits, wr)
    np.testing.assert_array_equal(logits, wr[:, cols].T)


@pytest.mark.parametrize("H,E,k,T", [(4096, 288, 8, 1024), (4096, 288, 8, 1500), (256, 16, 4, 2048),
                                     (768, 1000, 16, 1100), (512, 300, 6, 1030)])
def test_route_tensor_core_logits_match_oracle(H, E, k, T):
    """Tensor-core logits against the fp64 oracle.  Bound: the products are exact,
    so the error is the tensor core's fp32 accumulation (3 H / 16 steps of 16
    products; measured 1.7e-6 of sum |x w| at H 4096); 1e-5 of sum |x w| is about
    6x that and ~200x below the error of a lost second weight part (2^-9 of each
    weight); a lost third part is caught bit-exactly by the one-hot test."""
    x_bits = synthetic.activations_bits(T, H, seed=5)
    wr = synthetic.router_weights(E, H, seed=5)
    idx, w, logits = _route_with_logits(H, E, k, T, x_bits, wr)
    x = omoe.bf16_bits_to_f64(x_bits)
    ref = x @ wr.astype(np.float64).T
    scale = np.abs(x) @ np.abs(wr.astype(np.float64)).T
    ratio = np.max(np.abs(logits - ref) / np.maximum(scale, 1e-30))
    print(f"max |logit error| / sum|x w| = {ratio:.3e}")
    assert ratio < 1e-5
    near = check_routing(idx, w, omoe.route(x, wr, None, k))
    assert near <= max(1, T // 500)
