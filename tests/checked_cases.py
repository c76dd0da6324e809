"""A dispatch layout that a caller has overwritten with rows outside [0, R_max), run through every
entry point that reads it (imported by test_gpu_checked.py, in-process for the default build and
in a child process for the bounds-checked one).

Every kernel checks each row it reads from row_of, and the shared group's base
row_offsets[E] + t, against [0, R_max) before using it, in both builds, so the bad rows are
skipped. The padded-layout fill, which trusts row_offsets in the default build, is not run:
the layout is unpadded.  Each output buffer carries guard rows past R_max that must stay
untouched."""
import numpy as np
import torch

GUARD = 8


def run_corrupted_rows(ep) -> dict:
    T, K, E, H = 300, 4, 16, 256
    rng = np.random.default_rng(77)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    probs = torch.from_numpy(rng.random((T, K)).astype(np.float32)).cuda()
    L = ep.dispatch_layout(torch.from_numpy(ids).cuda(), E, fused_shared=True)
    assert ep.read_status(L) == 0
    R_max = L.R_max
    L.row_of[5, 2] = R_max + 7           # rows a caller wrote over the layout's own
    L.row_of[9, 0] = 1 << 30
    L.row_of[11, 1] = -5
    L.row_offsets[E] = R_max - 10        # the shared rows of tokens 10.. fall past R_max

    def guarded(cols, dtype, fill):
        return torch.full((R_max + GUARD, cols), fill, dtype=dtype, device="cuda")

    fp4, sc = guarded(H // 2, torch.uint8, 0x5A), guarded(H // 16, torch.uint8, 0x5A)
    inv = torch.full((R_max + GUARD,), 0x1357, dtype=torch.int16, device="cuda")
    so = torch.empty(E + 2, dtype=torch.int32, device="cuda")
    rows = guarded(H, torch.int16, 0x2468)
    f8 = guarded(H, torch.uint8, 0x5A)
    f8s = guarded(H // 128, torch.float32, 7.0)
    gy = guarded(H, torch.int16, 0x2468)
    y = torch.randn(R_max, H, device="cuda").to(torch.bfloat16)
    g = torch.randn(T, H, device="cuda").to(torch.bfloat16)

    ep.dispatch_nvfp4(x, L, out=(fp4[:R_max], sc[:R_max], inv[:R_max].view(torch.bfloat16), so))
    ep.dispatch_bf16(x, L, out=rows[:R_max].view(torch.bfloat16))
    ep.dispatch_fp8(x, L, out=(f8[:R_max], f8s[:R_max]))
    # (pre-zeroed: once the checked build has set its status bit, later calls write nothing)
    out = ep.combine(y, probs, L, out=torch.zeros(T, H, dtype=torch.bfloat16, device="cuda"))
    ep.combine_bwd(g, y, probs, L, out=(gy[:R_max].view(torch.bfloat16),
                                        torch.zeros(T, K, dtype=torch.float32, device="cuda")))
    gx = ep.dispatch_bwd(y, L, out=torch.zeros(T, H, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    guards = [bool((fp4[R_max:] == 0x5A).all()), bool((sc[R_max:] == 0x5A).all()),
              bool((inv[R_max:] == 0x1357).all()), bool((rows[R_max:] == 0x2468).all()),
              bool((f8[R_max:] == 0x5A).all()), bool((f8s[R_max:] == 7.0).all()),
              bool((gy[R_max:] == 0x2468).all())]
    status = ep.read_status(L)
    host = ctypes_status(ep, L)
    return {"checked": bool(ep.CHECKED), "lib": ep.LIB_PATH, "status": status, "read_status_rc": host,
            "guards_untouched": all(guards), "outputs_finite": bool(torch.isfinite(out.float()).all()
                                                                    and torch.isfinite(gx.float()).all())}


def ctypes_status(ep, L) -> int:
    import ctypes
    return int(ep.lib().ep_read_status(L.ref, None, ctypes.byref(ctypes.c_int32())))
