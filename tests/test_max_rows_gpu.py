"""The largest packed batch the ABI accepts: rows = 2^31 - 1 (cu_seqlens is
int32), C = 8, forward and backward (about 137 GB on the device).

Row indices then sit at the int32 limit, so every sum of a row index and a
small offset in the kernels (the next batch of the backward's copy ring,
the end of a walk, the prefetch row, the final-state rows, the step index
past a sequence's end that carries d_final_state) must be computed without
overflow.  The oracle cannot take the whole batch, so it checks windows:
every small sequence at the very end of the rows in full, and 2048-row
windows at the start and end of the long sequences, each with its three
history rows given as an initial state (FlashInfer causal_conv1d_fn,
Parameters: has_initial_state reads positions 0:3).  The weight and bias
gradients, sums over all 2^31 - 1 rows, are checked for bitwise
reproducibility instead.
"""
import numpy as np
import pytest
import torch

import oracle
import ssm_depthwise_causal_gb300 as ccc
from ssm_depthwise_causal_gb300 import workloads
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

ROWS = 2 ** 31 - 1
C = 8
WIN = 2048


def _window(x, dy, out, dx, weight, bias, s, e, hist, *, seq_end, d_final=None, what):
    """Rows [s, e) of one sequence against the oracle, history `hist` (3 BF16
    rows [3, C]) before s; dx is compared on every row only when e is the
    sequence's end (else the last 3 rows also depend on rows after e)."""
    xs = x[s:e].cpu()
    pool = hist.t().contiguous().view(1, C, 3)
    pool = torch.cat([pool, torch.zeros((1, C, 1), dtype=torch.bfloat16)], dim=2)
    cu = torch.tensor([0, e - s], dtype=torch.int32)
    ref_out, _, ref_hist = oracle.fwd(xs, weight.cpu(), bias.cpu(), cu, pool, torch.zeros(1, dtype=torch.int32),
                                      torch.ones(1, dtype=torch.bool))
    H.assert_bf16_close(H.bits(out[s:e]), ref_out, f"{what}: out")
    ref = oracle.bwd(xs, weight.cpu(), bias.cpu(), cu, dy[s:e].cpu(), ref_hist, torch.zeros(1, dtype=torch.int32),
                     torch.ones(1, dtype=torch.bool), None if d_final is None else d_final.cpu())
    n = e - s if seq_end else e - s - 3
    H.assert_bf16_close(H.bits(dx[s:s + n]), ref["dx"][:n], f"{what}: dx")
    return ref


def test_rows_at_the_int32_limit(cuda_device):
    dev = cuda_device
    if torch.cuda.get_device_properties(dev).total_memory < 200 * 10 ** 9:
        pytest.skip("needs ~140 GB of device memory")
    torch.cuda.empty_cache()  # blocks cached by earlier tests in this process
    g = workloads._gen(2024, dev)
    x = dy = out = dx = None
    try:
        x = workloads.normal_bf16((ROWS, C), g, dev, chunk_rows=1 << 24)
        dy = workloads.normal_bf16((ROWS, C), g, dev, chunk_rows=1 << 24)
        out = torch.empty_like(x)
        dx = torch.empty_like(x)
        weight = workloads.uniform((C, 4), g, dev, -0.5, 0.5, torch.float32)
        bias = (torch.randn((C,), generator=g, device=dev) * 0.1).to(torch.bfloat16)
        ws = torch.empty(ccc.ccc_workspace_size(ROWS, 8, C, True), dtype=torch.uint8, device=dev)

        # ---- eight sequences, the last six short and ending at row 2^31 - 1
        tail = [300, 5, 0, 1, 2, 700]
        a_len = 2 ** 30 + 12345
        lengths = np.array([a_len, ROWS - a_len - sum(tail)] + tail, dtype=np.int64)
        N = len(lengths)
        cu_np = np.concatenate([[0], np.cumsum(lengths)])
        assert cu_np[-1] == ROWS
        cu = torch.from_numpy(cu_np.astype(np.int32)).to(dev)
        cache = torch.tensor([3, 0, 5, 1, 6, -1, 2, 7], dtype=torch.int32, device=dev)
        hi = torch.tensor([1, 0, 1, 1, 0, 1, 1, 1], dtype=torch.bool, device=dev)
        pool = workloads.normal_bf16((8, C, 4), g, dev)
        pool0 = pool.cpu()
        hist = H.fill_sentinel(torch.empty((N, 3, C), dtype=torch.bfloat16, device=dev))
        dw = torch.empty((C, 4), device=dev)
        db = torch.empty((C,), device=dev)
        d_init = torch.empty((N, 3, C), device=dev)
        ccc.ccc_fwd(x, weight, bias, pool, cu, cache, hi, out, hist)
        ccc.ccc_bwd(x, weight, bias, hist, cu, cache, hi, dy, None, dx, dw, db, d_init, ws)
        dw1, db1 = dw.clone(), db.clone()
        ccc.ccc_bwd(x, weight, bias, hist, cu, cache, hi, dy, None, dx, dw, db, d_init, ws)
        torch.cuda.synchronize()
        assert torch.equal(dw, dw1) and torch.equal(db, db1), "dweight / dbias not reproducible"
        assert torch.isfinite(dw).all() and torch.isfinite(db).all()

        # the short sequences at the end, whole, with their own slots and flags
        s2 = int(cu_np[2])
        sub_cu = torch.from_numpy((cu_np[2:] - s2).astype(np.int32))
        xs, dys = x[s2:].cpu(), dy[s2:].cpu()
        ref_out, ref_state, ref_hist = oracle.fwd(xs, weight.cpu(), bias.cpu(), sub_cu, pool0, cache[2:].cpu(),
                                                  hi[2:].cpu())
        live = np.concatenate([np.full(n, c != -1) for n, c in zip(lengths[2:], cache[2:].tolist())])
        H.assert_bf16_close(H.bits(out[s2:])[live], ref_out[live], "tail: out")
        assert np.all(H.bits(out[s2:])[~live] == 0), "tail: -1 rows of out must be +0"
        ne = lengths[2:] > 0
        np.testing.assert_array_equal(H.bits(hist[2:])[ne], ref_hist[ne], err_msg="tail: saved_hist")
        ref = oracle.bwd(xs, weight.cpu(), bias.cpu(), sub_cu, dys, ref_hist, cache[2:].cpu(), hi[2:].cpu())
        H.assert_bf16_close(H.bits(dx[s2:])[live], ref["dx"][live], "tail: dx")
        assert np.all(H.bits(dx[s2:])[~live] == 0), "tail: -1 rows of dx must be +0"
        di, rdi = d_init[2:].cpu().double().numpy(), ref["d_init"]
        assert (np.abs(di - rdi) <= 1e-4 * np.abs(rdi) + 1e-5).all(), "tail: d_init_state"
        # every slot: the tail sequences' slots as the oracle left them, the
        # long sequences' slots hold their last three rows, the others untouched
        st = H.bits(pool)
        for n in range(2, N):
            q = int(cache[n])
            if q >= 0:
                np.testing.assert_array_equal(st[q], ref_state[q], err_msg=f"slot {q}")
        for n in range(2):
            q, e = int(cache[n]), int(cu_np[n + 1])
            np.testing.assert_array_equal(st[q, :, :3], H.bits(x[e - 3:e]).T, err_msg=f"slot {q}")
            np.testing.assert_array_equal(st[q, :, 3], H.bits(pool0)[q, :, 3], err_msg=f"slot {q} position 3")
        np.testing.assert_array_equal(st[4], H.bits(pool0)[4], err_msg="unused slot 4")

        # windows at the start and the end of the two long sequences
        for n in range(2):
            s, e = int(cu_np[n]), int(cu_np[n + 1])
            init = pool0[int(cache[n]), :, :3].t().contiguous() if bool(hi[n]) else torch.zeros((3, C), dtype=torch.bfloat16)
            ref = _window(x, dy, out, dx, weight, bias, s, s + WIN, init, seq_end=False, what=f"seq {n} start")
            di, rdi = d_init[n].cpu().double().numpy(), ref["d_init"][0]
            if not bool(hi[n]):
                rdi = np.zeros_like(rdi)
            assert (np.abs(di - rdi) <= 1e-4 * np.abs(rdi) + 1e-5).all(), f"seq {n}: d_init_state"
            _window(x, dy, out, dx, weight, bias, e - WIN, e, x[e - WIN - 3:e - WIN].cpu(), seq_end=True,
                    what=f"seq {n} end")

        # ---- one sequence of 2^31 - 1 rows, no pool, a d_final_state carried in
        cu1 = torch.tensor([0, ROWS], dtype=torch.int32, device=dev)
        d_final = torch.randn((1, 3, C), generator=g, device=dev)
        ccc.ccc_fwd(x, weight, bias, None, cu1, None, None, out)
        ccc.ccc_bwd(x, weight, bias, None, cu1, None, None, dy, d_final, dx, dw, db, d_init[:1], ws)
        torch.cuda.synchronize()
        zero = torch.zeros((3, C), dtype=torch.bfloat16)
        _window(x, dy, out, dx, weight, bias, 0, WIN, zero, seq_end=False, what="one sequence: start")
        mid = 2 ** 30 + 777
        _window(x, dy, out, dx, weight, bias, mid, mid + WIN, x[mid - 3:mid].cpu(), seq_end=False,
                what="one sequence: middle")
        _window(x, dy, out, dx, weight, bias, ROWS - WIN, ROWS, x[ROWS - WIN - 3:ROWS - WIN].cpu(), seq_end=True,
                d_final=d_final, what="one sequence: end")
    finally:
        del x, dy, out, dx
        torch.cuda.empty_cache()
