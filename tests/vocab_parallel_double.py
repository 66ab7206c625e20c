"""A CPU stand-in, in float64, for the library's per-shard steps of the
vocabulary-parallel JSD (``vpd_jsd_shard_*`` and the shard backward), with the
same buffer contract, so that the exchange protocol of
``softmax_divergence_lm_gb300.vocab_parallel`` (which all-reduce, with which
operation, in which order, between which steps) can run as gloo ranks on a
host without a GPU. Test infrastructure only; the row statistics come from the
oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import oracle as O


class NumpyShardKernels:
    def stats(self, s, t, saved, xbuf):
        for col, x in ((0, s), (2, t)):
            x64 = x.double().numpy()
            if x64.shape[1] == 0:
                m = np.full(x64.shape[0], -np.inf)
                lse = np.full(x64.shape[0], -np.inf)
            else:
                m, lse, code = O.row_stats(x64)
                m = np.where(code == 1, np.nan, np.where(code == 2, -np.inf, m))
                lse = np.where(code == 1, np.nan, np.where(code == 2, -np.inf, lse))
            saved[:, col] = torch.from_numpy(m)
            saved[:, col + 1] = torch.from_numpy(lse)
            xbuf[:, col // 2] = torch.from_numpy(np.where(np.isnan(m), np.inf, m))

    def rescale(self, rows, saved, xbuf):
        for h in range(2):
            ml, L, mg = saved[:, 2 * h].clone(), saved[:, 2 * h + 1].clone(), xbuf[:, h].clone()
            z = torch.where(ml == -math.inf, torch.zeros_like(ml), torch.exp(L + (ml - mg)))
            z = torch.where(torch.isnan(mg) | (mg == math.inf), torch.full_like(z, math.nan), z)
            saved[:, 2 * h] = mg
            xbuf[:, h] = z

    def _lse(self, saved, xbuf):
        for h in range(2):
            mg, Z = saved[:, 2 * h].clone(), xbuf[:, h].clone()
            bad = torch.isnan(Z) | torch.isnan(mg) | (mg == math.inf)
            L = torch.where(mg == -math.inf, torch.full_like(Z, -math.inf), torch.log(Z))
            saved[:, 2 * h] = torch.where(bad, torch.full_like(mg, math.nan), mg)
            saved[:, 2 * h + 1] = torch.where(bad, torch.full_like(L, math.nan), L)

    @staticmethod
    def _logp(x, m, L):
        x = x.double().numpy()
        with np.errstate(invalid="ignore"):
            return np.where(np.isneginf(x), -np.inf, (x - m[:, None]) - L[:, None])

    def divergence(self, s, t, beta, loss, saved, xbuf):
        self._lse(saved, xbuf)
        sv = saved.double().numpy()
        lp, lq = self._logp(s, sv[:, 0], sv[:, 1]), self._logp(t, sv[:, 2], sv[:, 3])
        fs, ft = np.isfinite(lp), np.isfinite(lq)
        p, q = np.where(fs, np.exp(np.where(fs, lp, 0)), 0), np.where(ft, np.exp(np.where(ft, lq, 0)), 0)
        with np.errstate(divide="ignore", invalid="ignore"):
            if 0.0 < beta < 1.0:
                lm = np.logaddexp(math.log(1 - beta) + lp, math.log(beta) + lq)
                A = np.sum(np.where(ft, q * (lq - lm), 0), axis=1)
                B = np.sum(np.where(fs, p * (lp - lm), 0), axis=1)
            elif beta == 0.0:
                A = np.sum(np.where(ft & fs, q * (lq - lp), 0), axis=1)
                A = np.where(np.any(ft & ~fs, axis=1), np.inf, A)
                B = np.zeros_like(A)
            else:
                B = np.sum(np.where(fs & ft, p * (lp - lq), 0), axis=1)
                B = np.where(np.any(fs & ~ft, axis=1), np.inf, B)
                A = np.zeros_like(B)
        ok = np.isfinite(sv[:, 0]) & np.isfinite(sv[:, 2])
        A, B = np.where(ok, A, np.nan), np.where(ok, B, np.nan)
        xbuf[:, 0], xbuf[:, 1] = torch.from_numpy(A), torch.from_numpy(B)
        loss[:] = torch.from_numpy(np.where(ok, beta * A + (1 - beta) * B, np.nan))

    def finish(self, rows, beta, saved, xbuf, loss):
        A, B = xbuf[:, 0].clone(), xbuf[:, 1].clone()
        ok = torch.isfinite(saved[:, 0]) & torch.isfinite(saved[:, 2])
        value = beta * A + (1 - beta) * B if 0.0 < beta < 1.0 else (A if beta == 0.0 else B)
        nan = torch.full_like(A, math.nan)
        saved[:, 4], saved[:, 5] = torch.where(ok, A, nan), torch.where(ok, B, nan)
        loss[:] = torch.where(ok, value, nan)

    def backward(self, s, t, beta, grad, saved, ds, dt):
        sv = saved.double().numpy()
        g = np.ones(sv.shape[0]) if grad is None else grad.double().numpy()
        lp, lq = self._logp(s, sv[:, 0], sv[:, 1]), self._logp(t, sv[:, 2], sv[:, 3])
        fs, ft = np.isfinite(lp), np.isfinite(lq)
        p, q = np.where(fs, np.exp(np.where(fs, lp, 0)), 0), np.where(ft, np.exp(np.where(ft, lq, 0)), 0)
        A, B = sv[:, 4:5], sv[:, 5:6]
        gg = g[:, None]
        with np.errstate(divide="ignore", invalid="ignore"):
            if 0.0 < beta < 1.0:
                lm = np.logaddexp(math.log(1 - beta) + lp, math.log(beta) + lq)
                gs = np.where(fs, gg * (1 - beta) * p * (lp - lm - B), 0)
                gt = np.where(ft, gg * beta * q * (lq - lm - A), 0)
            elif beta == 0.0:
                gs = gg * (p - q)
                gt = np.where(ft, gg * q * (lq - lp - A), 0)
            else:
                gs = np.where(fs, gg * p * (lp - lq - B), 0)
                gt = gg * (q - p)
        live = np.isfinite(sv[:, 0]) & np.isfinite(sv[:, 2]) & np.isfinite(sv[:, 4]) & np.isfinite(sv[:, 5])
        if ds is not None:
            ds[:] = torch.from_numpy(np.where(live[:, None], gs, 0.0))
        if dt is not None:
            dt[:] = torch.from_numpy(np.where(live[:, None], gt, 0.0))
