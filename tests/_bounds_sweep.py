"""The option sweep run by test_gpu_debug_bounds.py in a child process
against the bounds-checking debug build (KVQ_LIB_PATH): prefill, single-token
appends across window flushes, decode attention and dequant for every option
of the descriptor; every call must leave the status word at 0, and the blocks
and attention must match the oracle.  Not a test module itself."""

import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from bit_kv_cache_02_gb300 import kvq  # noqa: E402

LENS = [1, 31, 33, 127, 129, 255, 257]
ATOL, RTOL = 2e-3, 1e-2


def main():
    assert kvq.LIB_PATH == os.environ["KVQ_LIB_PATH"], "not the debug build"
    rng = np.random.default_rng(3)
    S, H, gq, T = len(LENS), 2, 2, max(LENS)
    cases = [dict(), dict(pre_rope=True), dict(kpt=True), dict(rot=True), dict(sp=True), dict(paged=True)]
    n = 0
    for bits in (2, 4):
        for ns in (0, 1):
            for c in cases:
                pre_rope, kpt, rot, sp, paged = (c.get(x, False) for x in ("pre_rope", "kpt", "rot", "sp", "paged"))
                cap = T + 8
                cache = kvq.KVCache(S, H, cap, bits=bits, num_sink=ns, pre_rope=pre_rope, key_per_token=kpt,
                                    hadamard=rot, outliers=sp, paged=paged)
                if paged:
                    perm = rng.permutation(cache.num_blocks).astype(np.int32)
                    cache.block_table.copy_(torch.from_numpy(perm.reshape(cache.block_table.shape)).cuda())
                orc = oracle.OracleCache(S, H, cap, bits, num_sink=ns, key_per_token=kpt, hadamard=rot, outliers=sp)
                k = (rng.standard_normal((S, H, T, 128)) * 2).astype(np.float16)
                v = rng.standard_normal((S, H, T, 128)).astype(np.float16)
                pre = [max(L - 3, 0) for L in LENS]
                kvq.kv_quant_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                                    torch.tensor(pre, dtype=torch.int32).cuda(), T)
                orc.append(k, v, pre)
                for step in range(3):  # single-token appends (the fused step kernel)
                    lens = [1 if pre[s] + step < LENS[s] else 0 for s in range(S)]
                    idx = [min(pre[s] + step, T - 1) for s in range(S)]
                    k1 = np.stack([k[s, :, idx[s]:idx[s] + 1] for s in range(S)])
                    v1 = np.stack([v[s, :, idx[s]:idx[s] + 1] for s in range(S)])
                    kvq.kv_quant_append(cache, torch.from_numpy(np.ascontiguousarray(k1)).cuda(),
                                        torch.from_numpy(np.ascontiguousarray(v1)).cuda(),
                                        torch.tensor(lens, dtype=torch.int32).cuda(), 1)
                    orc.append(k1, v1, lens)
                q = rng.standard_normal((S, H * gq, 128)).astype(np.float16)
                dq = torch.from_numpy(q).cuda()
                out = torch.empty_like(dq)
                ws = kvq.alloc_workspace(cache, H * gq, T)
                kvq.kv_decode_attn(cache, dq, out, ws, T)
                K = torch.empty((S, H, cap, 128), device="cuda")
                V = torch.empty_like(K)
                kvq.kv_dequant(cache, K, V)
                torch.cuda.synchronize()
                st = int(cache.status.item())
                assert st == 0, f"status {st} with bits={bits} ns={ns} {c}"
                got = out.cpu().numpy().astype(np.float64)
                want = orc.attention(q, pre_rope=pre_rope).astype(np.float64)
                err = np.abs(got - want)
                assert (err <= ATOL + RTOL * np.abs(want)).all(), f"attention, bits={bits} ns={ns} {c}: {err.max()}"
                blocks = cache.logical_blocks().cpu().numpy()
                for s in range(S):
                    ng = orc.split(s)[1] // 32
                    np.testing.assert_array_equal(blocks[s, :, :ng], orc.blocks[s, :, :ng])
                n += 1
    print(f"bounds sweep ok: {n} caches")


if __name__ == "__main__":
    main()
