"""Host logic of the launch plan (moe_plan: no GPU needed): the decode/prefill switch,
K splits that divide the K chunks, grids sized in whole waves of the SM count, the
fused small-batch routing condition and a row-chunk capacity that covers any routing."""
import pytest

import routed_expert_layer_gb300 as rel

K3 = dict(hidden=7168, inter=1536, n_experts=896, top_k=16)
SM = 152


def plan(T, max_tokens=8192, sm=SM, **shape):
    s = dict(K3)
    s.update(shape)
    return rel.plan(s["hidden"], s["inter"], s["n_experts"], s["top_k"], max_tokens, sm, T)


@pytest.mark.parametrize("T", [1, 2, 8, 32, 33, 53, 64, 128, 256, 447, 448, 1024, 2048, 2239, 2240, 4096, 5375,
                               5376, 8192])
def test_k3_plans(T):
    p = plan(T)
    H, I, E, k = K3["hidden"], K3["inter"], K3["n_experts"], K3["top_k"]
    prefill = T * k / E >= 8
    assert p["prefill"] == int(prefill)
    # decode: 16-row items; midfill: 64 below 40 rows per expert on average, 128 below 96;
    # prefill: 192
    avg = T * k / E
    assert p["rows_per_item"] == (16 if not prefill else (64 if avg < 40 else (128 if avg < 96 else 192)))
    # prefill-sized calls on the general routing path send experts of at most 16 rows to
    # the decode GEMM
    assert p["cold_rows"] == (16 if prefill and not p["fused_routing"] else 0)
    assert p["gemm_ctas"] == (SM if prefill else 2 * SM)
    for key, kc in (("gateup_splits", H // 128), ("down_splits", I // 128)):
        s = p[key]
        assert kc % s == 0 and (s == 1 or s <= kc // 3)
        if prefill:
            assert s == 1
    kc_router = 3 * H // 64
    assert kc_router % p["router_splits"] == 0
    assert 1 <= p["router_ctas"] <= SM
    assert p["fused_routing"] == int(T <= 32)
    # any routing yields at most min(E, T*k) + T*k / rows_per_item + 1 row chunks
    rows = T * k
    assert p["chunk_capacity"] >= min(E, rows) + rows // p["rows_per_item"] + 1


def test_capacity_covers_every_batch_size_up_to_max_tokens():
    cap = plan(1, max_tokens=512)["chunk_capacity"]
    for T in range(1, 513, 7):
        p = plan(T, max_tokens=512)
        rows = T * K3["top_k"]
        assert cap >= min(K3["n_experts"], rows) + rows // p["rows_per_item"] + 1


def test_fused_routing_needs_few_router_splits():
    # one 128-expert router tile and a wide K: the splits exceed what the fused kernel stages
    p = plan(1, hidden=14336, inter=256, n_experts=16, top_k=4, max_tokens=64)
    assert p["router_splits"] > 64 and p["fused_routing"] == 0
    # E not a multiple of 4
    assert plan(1, hidden=256, inter=128, n_experts=1, top_k=1, max_tokens=64)["fused_routing"] == 0


def test_workspace_grows_with_max_tokens():
    assert plan(1, max_tokens=64)["workspace_bytes"] < plan(1, max_tokens=8192)["workspace_bytes"]


def test_plan_rejects_bad_arguments():
    with pytest.raises(rel.MoeError) as ei:
        plan(0)
    assert ei.value.status == rel.MOE_ERR_INVALID_ARG
    with pytest.raises(rel.MoeError):
        plan(9000)
    with pytest.raises(rel.MoeError):
        plan(1, sm=0)
    with pytest.raises(rel.MoeError) as ei:
        plan(1, hidden=7000)
    assert ei.value.status == rel.MOE_ERR_UNSUPPORTED
