"""The time-sharded forward's exchange (``tsplit.forward_time_sharded``) on gloo
ranks on CPU: each rank holds consecutive tokens of the same sequences, the
three steps are done by the fp64 oracle, and every rank's shard must equal the
same tokens of one unsharded oracle run (slide 9: the natural-parameter
recurrences are affine in the state, so shard summaries compose in order)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_ops():
    import oracle
    from metaplastic_linear_attention_gb300.tsplit import ShardOps

    n = lambda t: None if t is None else t.numpy()

    def summary(q, k, v, beta, d_t, A, Ip):
        B, H, T, dk = q.shape
        dv = v.shape[-1]
        if T == 0:
            return torch.zeros((B, H, 2, dv, dk), dtype=torch.float64), torch.ones((B, H), dtype=torch.float64)
        _, mu, I = oracle.forward(n(q), n(k), n(v), n(beta), n(d_t), n(A), n(Ip))   # zero excess state
        Ipg = n(Ip)[None, :, None, None]
        s = np.stack([mu * I, I - Ipg], axis=2)
        gamma = np.exp(-n(A)[None, :] * n(d_t).sum(-1))                            # product of the alphas
        return torch.from_numpy(s), torch.from_numpy(gamma)

    def combine(S, G, Ip, mu0, I0):
        Ipg = n(Ip)[None, :, None, None]
        shape = mu0.shape if mu0 is not None else (S.shape[1], S.shape[2], S.shape[4], S.shape[5])
        i0 = n(I0) if I0 is not None else np.broadcast_to(Ipg, shape).copy()
        m = i0 * (n(mu0) if mu0 is not None else 0.0)
        ib = i0 - Ipg
        for s in range(S.shape[0]):
            g = n(G[s])[..., None, None]
            m = g * m + n(S[s])[:, :, 0]
            ib = g * ib + n(S[s])[:, :, 1]
        I = Ipg + ib
        return torch.from_numpy(m / I), torch.from_numpy(I)

    def forward(q, k, v, beta, d_t, A, Ip, mu0, I0):
        return tuple(torch.from_numpy(x) for x in
                     oracle.forward(n(q), n(k), n(v), n(beta), n(d_t), n(A), n(Ip), mu0=n(mu0), I0=n(I0)))

    return ShardOps(summary=summary, combine=combine, forward=forward)


def _problem(seed, B=1, H=2, T=60, dk=6, dv=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T, dv))))
    d_t = np.log1p(np.exp(rng.standard_normal((B, H, T))))
    A = rng.uniform(0.1, 1.0, H)
    Ip = rng.uniform(0.5, 2.0, H)
    mu0 = rng.standard_normal((B, H, dv, dk))
    I0 = rng.uniform(0.5, 3.0, (B, H, dv, dk))
    return q, k, v, beta, d_t, A, Ip, mu0, I0


def _rank_main(rank, ws, port, bounds, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        from metaplastic_linear_attention_gb300.tsplit import forward_time_sharded
        q, k, v, beta, d_t, A, Ip, mu0, I0 = (torch.from_numpy(x) for x in _problem(7))
        t0, t1 = bounds[rank], bounds[rank + 1]
        sl = lambda x: x[:, :, t0:t1].contiguous()
        y, mu, I = forward_time_sharded(sl(q), sl(k), sl(v), sl(beta), sl(d_t), A, Ip, mu0, I0,
                                        ops=_oracle_ops())
        out[rank] = (y.numpy(), mu.numpy(), I.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bounds", [[0, 25, 60], [0, 13, 13, 60]], ids=["two_ranks", "three_ranks_one_empty"])
def test_time_sharded_forward_equals_one_pass(bounds):
    import oracle
    ws = len(bounds) - 1
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(ws, _free_port(), bounds, out), nprocs=ws, start_method="spawn", join=True)
    q, k, v, beta, d_t, A, Ip, mu0, I0 = _problem(7)
    y_ref, mu_ref, I_ref = oracle.forward(q, k, v, beta, d_t, A, Ip, mu0=mu0, I0=I0)
    for r in range(ws):
        y, mu, I = out[r]
        np.testing.assert_allclose(y, y_ref[:, :, bounds[r]:bounds[r + 1]], rtol=1e-10, atol=1e-12)
        # the state at the end of shard r is the one-pass state after token bounds[r + 1]
        _, mu_r, I_r = oracle.forward(q[:, :, :bounds[r + 1]], k[:, :, :bounds[r + 1]], v[:, :, :bounds[r + 1]],
                                      beta[:, :, :bounds[r + 1]], d_t[:, :, :bounds[r + 1]], A, Ip, mu0=mu0, I0=I0)
        np.testing.assert_allclose(mu, mu_r, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(I, I_r, rtol=1e-12)
    np.testing.assert_allclose(out[ws - 1][1], mu_ref, rtol=1e-10, atol=1e-12)
