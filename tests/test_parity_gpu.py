"""CUDA path vs the float64 oracle on small cases that span several 64-token
blocks and ragged tails (GPU).  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import mla_harness as Hn
import mla_inputs as I
import mla_latent_kv_81_b300 as M
from gpu_helpers import assert_close, oracle_sequence
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"
# DeepSeek-V2 head shapes with a small model width (keeps the oracle's weights small)
DSV2_NARROW = I.Dims(d_model=512, n_heads=128, qk_nope=128, d_rope=64, v_head=128, d_c=512)


def _status_clean(L):
    code, flags = L.status()
    assert code == 0, (M.mla_status_string(code), flags)


def test_tiny_f32_end_to_end():
    """The tiny fp32 layer: cache built by append, one query, every stage and the output."""
    p = I.make_problem(I.WORKLOADS["tiny_f32_b1_ctx10"])
    L = Hn.DeviceLayer(p)
    L.fill()
    L.step()
    torch.cuda.synchronize()
    _status_clean(L)
    ref = oracle_sequence(p, 0)
    rows = L.cache_rows_logical(0)
    assert_close(rows[:, :p.dims.d_c], ref["c"], "f32", "c")
    assert_close(rows[:, p.dims.d_c:], ref["k_r"], "f32", "k_R")
    q = L.q.cpu().numpy()
    assert_close(q[..., :p.dims.d_c], ref["q_abs"], "f32", "q_abs")
    assert_close(q[..., p.dims.d_c:], ref["q_rope"], "f32", "q_R")
    assert_close(L.o_lat.cpu().numpy(), ref["o_lat"], "f32", "o_lat")
    assert_close(L.lse.cpu().numpy(), ref["lse"], "f32", "lse")
    assert_close(L.out.cpu().numpy(), ref["out"], "f32", "out")


def _stage_decode(dims, dtype, lens, n_q, seed, sharp=1.0, kv_extra=0):
    """Attention alone: drawn queries and drawn cache rows, checked per sequence."""
    w = I.Workload("stage", dims, dtype, len(lens), 1, 1, n_q, 0, seed, "direct")
    p = I.make_problem(w, with_weights=False, lens=lens)
    L = Hn.DeviceLayer.__new__(Hn.DeviceLayer)
    L.p, L.device, L.dt, L.cfg = p, DEV, Hn.tdtype(dtype), M.make_config(dims, dtype)
    L.pool = torch.full((p.num_blocks, dims.row, dims.block_size), float("nan"), dtype=L.dt, device=DEV)
    L.block_table = torch.from_numpy(p.block_table).to(DEV)
    L.cache = M.make_cache(L.pool, L.block_table, dims.block_size)
    L.kv_len = torch.from_numpy(p.kv_len.astype(np.int32)).to(DEV)
    L.ws = {}
    L.fill_direct()
    qn = I.draw_stage_query(dims, dtype, len(lens) * n_q, seed, sharp)
    q = Hn.to_dev(qn, dtype, DEV)
    L.o_lat = torch.empty((len(lens) * n_q, dims.n_heads, dims.d_c), dtype=L.dt, device=DEV)
    L.lse = torch.empty((len(lens) * n_q, dims.n_heads), dtype=torch.float32, device=DEV)
    L.attend(q=q)
    torch.cuda.synchronize()
    _status_clean(L)
    o = L.o_lat.float().cpu().numpy()
    lse = L.lse.cpu().numpy()
    scale = O.softmax_scale(dims.qk_nope, dims.d_rope)
    for b, n in enumerate(lens):
        rows = I.draw_latent_rows(w, b, int(n)).astype(np.float64)
        sl = slice(b * n_q, (b + 1) * n_q)
        ref_o, ref_lse = O.attend_latent(qn[sl, :, :dims.d_c], qn[sl, :, dims.d_c:], rows[:, :dims.d_c],
                                         rows[:, dims.d_c:], int(n), scale)
        seen = [j for j in range(n_q) if O.visible(int(n), n_q, j) > 0]
        for j in range(n_q):
            if j not in seen:
                assert np.all(o[b * n_q + j] == 0) and np.isneginf(lse[b * n_q + j]).all()
        if not seen:
            continue
        rows = [b * n_q + j for j in seen]
        assert_close(o[rows], ref_o[seen], dtype, f"o_lat[b={b}, L={n}]")
        assert np.all(np.abs(lse[rows] - ref_lse[seen]) <= 1e-3 * (1 + np.abs(ref_lse[seen]))), f"lse b={b}"


@pytest.mark.parametrize("n_q", [1, 2])
@pytest.mark.parametrize("sharp", [1.0, 8.0])
def test_decode_bf16_ragged(n_q, sharp):
    _stage_decode(I.DSV2, "bf16", [1, 63, 64, 65, 200, 1000, 4097], n_q, seed=21, sharp=sharp)


@pytest.mark.parametrize("lens", [
    [0, 1, 2],            # fewer tiles than clusters, one query with nothing visible
    [20000],              # one sequence split across every cluster
    [64] * 150,           # about two whole tiles per cluster
    [4096, 0, 17, 8191],  # mixed, with an empty sequence in the middle
])
def test_decode_bf16_split_regimes(lens):
    _stage_decode(I.DSV2, "bf16", lens, 1, seed=26)


def test_decode_f32_tiny_shapes_ragged():
    _stage_decode(I.TINY, "f32", [1, 10, 64, 65, 300], 1, seed=22)
    _stage_decode(I.TINY, "f32", [2, 10, 64, 65, 300], 2, seed=23)


def test_output_project_bf16():
    dims = DSV2_NARROW
    N = 37
    rng = np.random.default_rng(31)
    W = I.draw_weights(dims, "bf16", rng)
    o_lat = I.draw_stage_latent_out(dims, "bf16", N, 31)
    cfg = M.make_config(dims, "bf16")
    out = torch.empty((N, dims.d_model), dtype=torch.bfloat16, device=DEV)
    M.mla_output_project(cfg, Hn.to_dev(o_lat, "bf16"), Hn.to_dev(W["W_UV"], "bf16"), Hn.to_dev(W["W_O"], "bf16"),
                         out)
    ref = O.output_project(O.up_project_values(o_lat, W["W_UV"]), W["W_O"])
    assert_close(out.float().cpu().numpy(), ref, "bf16", "out")


def test_absorb_query_bf16():
    dims = DSV2_NARROW
    N = 37
    rng = np.random.default_rng(32)
    W = I.draw_weights(dims, "bf16", rng)
    x = I.draw_hidden(rng, N, dims.d_model, "bf16")
    q_pos = rng.integers(0, 70000, size=N).astype(np.int32)
    cfg = M.make_config(dims, "bf16")
    tab = torch.empty((70001, dims.d_rope // 2, 2), dtype=torch.float32, device=DEV)
    M.mla_rope_table_create(cfg, dims.rope_base, 70001, tab)
    q = torch.empty((N, dims.n_heads, dims.row), dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(M.mla_absorb_workspace_bytes(cfg, N), DEV)
    M.mla_absorb_query(cfg, Hn.to_dev(x, "bf16"), Hn.to_dev(W["W_Q"], "bf16"), Hn.to_dev(W["W_QR"], "bf16"),
                       Hn.to_dev(W["W_UK"], "bf16"), torch.from_numpy(q_pos).to(DEV), M.make_rope(tab), q, ws=ws)
    q_nope, q_rope = O.project_query(x, W["W_Q"], W["W_QR"], q_pos, dims.n_heads, dims.rope_base)
    q_abs = O.absorb_query(q_nope, W["W_UK"])
    got = q.float().cpu().numpy()
    assert_close(got[..., :dims.d_c], q_abs, "bf16", "q_abs")
    assert_close(got[..., dims.d_c:], q_rope, "bf16", "q_R")
    code, flags = M.mla_get_device_status(ws)
    assert code == 0, (M.mla_status_string(code), flags)


@pytest.mark.parametrize("n_q,n_append", [(1, 0), (2, 2), (1, 1)])
def test_end_to_end_bf16_narrow(n_q, n_append):
    """All steps chained through the ABI (append, absorb, attend, project) vs the explicit form."""
    w = I.Workload("e2e", DSV2_NARROW, "bf16", 3, 1, 1, n_q, n_append, 41 + n_q, "append")
    p = I.make_problem(w, lens=[5, 130, 700])
    L = Hn.DeviceLayer(p)
    L.fill()
    L.step()
    torch.cuda.synchronize()
    _status_clean(L)
    out = L.out.float().cpu().numpy()
    o_lat = L.o_lat.float().cpu().numpy()
    for b in range(3):
        ref = oracle_sequence(p, b)
        sl = slice(b * n_q, (b + 1) * n_q)
        assert_close(o_lat[sl], ref["o_lat"], "bf16", f"o_lat b={b}")
        assert_close(out[sl], ref["out"], "bf16", f"out b={b}")


def test_device_index_errors_are_flagged_not_faulted():
    """Out-of-range positions / block ids are skipped and reported in the status word of the workspace
    the call used."""
    dims = I.TINY
    w = I.Workload("idx", dims, "f32", 2, 1, 1, 1, 0, 5, "append")
    p = I.make_problem(w, lens=[10, 70])
    L = Hn.DeviceLayer(p)
    L.fill()
    torch.cuda.synchronize()
    _status_clean(L)
    before = L.pool.clone()
    cap = p.block_table.shape[1] * dims.block_size
    x = Hn.to_dev(p.x_q[:3], "f32")
    seq = torch.tensor([0, 5, 1], dtype=torch.int32, device=DEV)          # 5: outside the batch
    pos = torch.tensor([cap + 3, 2, -1], dtype=torch.int32, device=DEV)   # beyond blocks, fine, negative
    ws = M.workspace(M.mla_compress_workspace_bytes(L.cfg, 3), DEV)
    M.mla_compress_append(L.cfg, x, L.W["W_DKV"], L.W["W_KR"], seq, pos, L.rope, L.cache, ws=ws)
    code, flags = M.mla_get_device_status(ws)
    assert code == 5 and flags & 1
    assert M.mla_get_device_status(ws) == (0, 0)   # read and cleared
    assert torch.equal(torch.isnan(before), torch.isnan(L.pool))
    assert torch.equal(before.nan_to_num(7.0), L.pool.nan_to_num(7.0))
    # a kv_len beyond the table is clamped and flagged
    L.kv_len[1] = cap + 100
    L.q.copy_(Hn.to_dev(I.draw_stage_query(dims, "f32", 2, 5), "f32"))
    L.attend()
    code, flags = L.status()
    assert code == 5
    _status_clean(L)


def test_status_words_of_two_workspaces_on_two_streams_are_independent():
    """A flag raised by a call on one stream (its workspace) is not seen through another workspace used
    on another stream, and is cleared only by reading its own workspace."""
    dims = I.TINY
    w = I.Workload("two_streams", dims, "f32", 2, 1, 1, 1, 0, 6, "append")
    p = I.make_problem(w, lens=[10, 70])
    L = Hn.DeviceLayer(p)
    L.fill()
    torch.cuda.synchronize()
    _status_clean(L)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = M.workspace(M.mla_compress_workspace_bytes(L.cfg, 2), DEV)
    ws2 = M.workspace(M.mla_compress_workspace_bytes(L.cfg, 2), DEV)
    x = Hn.to_dev(p.x_q[:2], "f32")
    bad_pos = torch.tensor([-1, 3], dtype=torch.int32, device=DEV)
    good_pos = torch.tensor([70, 71], dtype=torch.int32, device=DEV)
    seq = torch.tensor([1, 1], dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        M.mla_compress_append(L.cfg, x, L.W["W_DKV"], L.W["W_KR"], seq, bad_pos, L.rope, L.cache, ws=ws1,
                              stream=s1)
    with torch.cuda.stream(s2):
        M.mla_compress_append(L.cfg, x, L.W["W_DKV"], L.W["W_KR"], seq, good_pos, L.rope, L.cache, ws=ws2,
                              stream=s2)
    assert M.mla_get_device_status(ws2, s2) == (0, 0)
    code, flags = M.mla_get_device_status(ws1, s1)
    assert code == 5 and flags == 1
    assert M.mla_get_device_status(None, s1) == (0, 0)   # the library's own word saw nothing


def test_bounded_wait_runs_out_and_reports_a_timeout():
    """Failure detection: a kernel whose wait is never satisfied gives up after its (short, test-only)
    limit, flags a timeout in the workspace's status word and returns; the context stays usable."""
    ws = M.workspace(256, DEV)
    M.mla_selftest_wait_timeout(ws, 2_000_000)   # ~1 ms of SM cycles
    code, flags = M.mla_get_device_status(ws)
    assert code == 4 and flags == 2
    assert M.mla_get_device_status(ws) == (0, 0)
    # the context still runs work afterwards
    t = torch.arange(1024, device=DEV, dtype=torch.float32)
    assert float(t.sum()) == 1023 * 1024 / 2


def test_bf16_shapes_outside_the_tensor_core_kernels_are_unsupported():
    """bf16 runs only on the tcgen05 kernels: a bf16 layer with other head shapes is refused by every
    entry point (no silent second backend); the same shapes in fp32 run."""
    dims = I.Dims(d_model=256, n_heads=16, qk_nope=32, d_rope=32, v_head=48, d_c=256)
    cfg = M.make_config(dims, "bf16")
    assert M.mla_decode_workspace_bytes(cfg, 2, 1, 4) == 0
    assert M.mla_absorb_workspace_bytes(cfg, 2) == 0
    assert M.mla_output_workspace_bytes(cfg, 2) == 0
    q = torch.zeros((2, dims.n_heads, dims.row), dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros((4, dims.row, dims.block_size), dtype=torch.bfloat16, device=DEV)
    table = torch.zeros((2, 2), dtype=torch.int32, device=DEV)
    kv = torch.ones(2, dtype=torch.int32, device=DEV)
    o = torch.zeros((2, dims.n_heads, dims.d_c), dtype=torch.bfloat16, device=DEV)
    ws = M.workspace(1 << 20, DEV)
    with pytest.raises(M.MlaError) as e:
        M.mla_decode_attention(cfg, q, M.make_cache(pool, table, dims.block_size), kv, 2, 1, o, ws=ws)
    assert e.value.code == 2
    _stage_decode(dims, "f32", [1, 64, 65, 300], 1, seed=24)
