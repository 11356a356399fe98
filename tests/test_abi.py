"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments with a status (no GPU needed:
validation runs before any device work)."""
import ctypes
import os
import re

import pytest
import torch

import momentum_delta_rule_gb300 as mdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mdn_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    from momentum_delta_rule_gb300 import build
    build.build()
    return mdn.lib()


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert set(declared) == set(mdn.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(L, name), name


def test_version_and_strings(L):
    assert mdn.abi_version() == 2
    for code in range(5):
        s = mdn.status_string(code)
        assert s.startswith("MDN")
    assert "unknown" in mdn.status_string(99)


def test_workspace_size(L):
    a = mdn.workspace_size(8, 16384, 8, 128, 1)
    assert a > 0 and a % 256 == 0
    assert mdn.workspace_size(-1, 10, 1, 64, 1) == 0
    assert mdn.workspace_size(1, 10, 1, 64, 7) == 0
    # monotone in the number of tokens and heads
    assert mdn.workspace_size(8, 16384, 16, 128, 1) > a


FAKE = ctypes.c_void_p(0x10000)       # a non-null pointer never dereferenced


def _chunk(L, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, mu=FAKE, eta=FAKE,
                beta=None, S0=None, M0=None, o=FAKE, S_T=None, M_T=None,
                cu=None, n_seq=2, B=2, T=64, H=2, dk=128, dv=128, dtype=1,
                chunk=64, ws=FAKE, ws_bytes=1 << 30, stream=None)
    args.update(over)
    return L.mdn_chunk_fwd(args["q"], args["k"], args["v"], args["alpha"],
                           args["mu"], args["eta"], args["beta"], args["S0"],
                           args["M0"], args["o"], args["S_T"], args["M_T"],
                           args["cu"], args["n_seq"], args["B"], args["T"],
                           args["H"], args["dk"], args["dv"], args["dtype"],
                           args["chunk"], args["ws"], args["ws_bytes"],
                           args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(alpha=None), 1), (dict(o=None), 1),
    (dict(H=0), 1), (dict(T=-1), 1), (dict(n_seq=3), 1), (dict(dtype=5), 1),
    (dict(q=ctypes.c_void_p(0x10008)), 1), (dict(ws=None), 1),
    (dict(ws_bytes=16), 1), (dict(ws=ctypes.c_void_p(0x10010)), 1),
    (dict(cu=FAKE, B=2), 1),
    (dict(S_T=FAKE, M_T=FAKE), 1),
    (dict(chunk=32), 2), (dict(dk=96, dv=96), 2), (dict(dk=128, dv=64), 2),
])
def test_chunk_fwd_rejects(L, over, code):
    assert _chunk(L, **over) == code


def _chunk_static(L, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, mu=FAKE, eta=FAKE,
                beta=None, S0=None, M0=None, o=FAKE, S_T=None, M_T=None,
                cu=None, n_seq=2, B=2, T=64, H=2, dk=128, dv=128, dtype=1,
                chunk=64, stream=None)
    args.update(over)
    return L.mdn_chunk_fwd_static_ws(args["q"], args["k"], args["v"], args["alpha"],
                                     args["mu"], args["eta"], args["beta"], args["S0"],
                                     args["M0"], args["o"], args["S_T"], args["M_T"],
                                     args["cu"], args["n_seq"], args["B"], args["T"],
                                     args["H"], args["dk"], args["dv"], args["dtype"],
                                     args["chunk"], args["stream"])


@pytest.mark.parametrize("over,code", [
    # the argument errors of mdn_chunk_fwd come first, even for problems whose
    # scratch would exceed the fixed array
    (dict(n_seq=1 << 24), 1), (dict(q=None), 1), (dict(dtype=5), 1),
    (dict(cu=FAKE, B=2), 1), (dict(S_T=FAKE, M_T=FAKE), 1),
    (dict(chunk=32), 2), (dict(dk=96, dv=96), 2),
    (dict(chunk=32, n_seq=1 << 24, B=1 << 24), 2),
])
def test_chunk_fwd_static_ws_rejects_like_chunk_fwd(L, over, code):
    assert _chunk_static(L, **over) == code


def _chunk_vres(L, vres, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, mu=FAKE, eta=FAKE,
                beta=None, S0=None, M0=None, o=FAKE, S_T=None, M_T=None,
                cu=None, n_seq=2, B=2, T=64, H=2, dk=128, dv=128, dtype=1,
                chunk=64, ws=FAKE, ws_bytes=1 << 30, stream=None)
    args.update(over)
    return L.mdn_chunk_fwd_vres(args["q"], args["k"], args["v"], args["alpha"],
                                args["mu"], args["eta"], args["beta"], args["S0"],
                                args["M0"], args["o"], args["S_T"], args["M_T"], vres,
                                args["cu"], args["n_seq"], args["B"], args["T"],
                                args["H"], args["dk"], args["dv"], args["dtype"],
                                args["chunk"], args["ws"], args["ws_bytes"],
                                args["stream"])


@pytest.mark.parametrize("vres,over,code", [
    (None, {}, 1),                                   # required when tokens exist
    (FAKE, {}, 1),                                   # aliases o (and q, k, v)
    (ctypes.c_void_p(0x30008), {}, 1),               # not 16-byte aligned
    (ctypes.c_void_p(0x30000), dict(chunk=32), 2),   # the rest as mdn_chunk_fwd
    (ctypes.c_void_p(0x30000), dict(q=None), 1),
])
def test_chunk_fwd_vres_rejects(L, vres, over, code):
    assert _chunk_vres(L, vres, **over) == code


def _prep(L, **over):
    args = dict(q=FAKE, k=ctypes.c_void_p(0x20000), za=FAKE, zb=FAKE, zm=FAKE, ze=FAKE,
                qo=ctypes.c_void_p(0x30000), ko=ctypes.c_void_p(0x40000), al=FAKE, be=FAKE,
                mu=FAKE, eta=FAKE, n=16, H=2, d=128, dtype=1, a=1.0, b=0.0, s=1.0,
                tau=1.0, lmin=-2.0, cd=0.0, stream=None)
    args.update(over)
    return L.mdn_prepare_inputs(args["q"], args["k"], args["za"], args["zb"], args["zm"],
                                args["ze"], args["qo"], args["ko"], args["al"], args["be"],
                                args["mu"], args["eta"], args["n"], args["H"], args["d"],
                                args["dtype"], args["a"], args["b"], args["s"], args["tau"],
                                args["lmin"], args["cd"], args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(q=None), 1), (dict(za=None), 1), (dict(eta=None), 1), (dict(n=-1), 1),
    (dict(H=0), 1), (dict(dtype=7), 1), (dict(a=0.0), 1), (dict(a=float("nan")), 1),
    (dict(tau=0.0), 1), (dict(qo=ctypes.c_void_p(0x30004)), 1),
    (dict(al=ctypes.c_void_p(0x10002)), 1), (dict(ko=ctypes.c_void_p(0x30000)), 1),
    (dict(qo=ctypes.c_void_p(0x20000)), 1), (dict(d=96), 2),
])
def test_prepare_inputs_rejects(L, over, code):
    assert _prep(L, **over) == code


def _decode(L, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, mu=FAKE, eta=FAKE,
                beta=None, S=FAKE, M=ctypes.c_void_p(0x20000), o=FAKE, N=4,
                H=2, dk=128, dv=128, dtype=1, stream=None)
    args.update(over)
    return L.mdn_decode_step(args["q"], args["k"], args["v"], args["alpha"],
                             args["mu"], args["eta"], args["beta"], args["S"],
                             args["M"], args["o"], args["N"], args["H"],
                             args["dk"], args["dv"], args["dtype"], args["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(S=None), 1), (dict(q=None), 1), (dict(N=-1), 1), (dict(H=0), 1),
    (dict(S=ctypes.c_void_p(0x10004)), 1), (dict(M=FAKE), 1),
    (dict(q=ctypes.c_void_p(0x10001)), 1), (dict(dtype=3), 1),
    (dict(dk=32, dv=32), 2), (dict(dk=64, dv=128), 2),
])
def test_decode_rejects(L, over, code):
    assert _decode(L, **over) == code


def test_binding_requires_cuda_tensors():
    import torch
    x = torch.zeros(1, 64, 1, 64)
    g = torch.zeros(1, 64, 1)
    with pytest.raises(ValueError):
        mdn.chunk_fwd(x, x, x, g, g, g)


def _chunk_states(L, Sc, Mc, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, mu=FAKE, eta=FAKE,
                beta=None, S0=None, M0=None, o=FAKE, S_T=None, M_T=None,
                cu=None, n_seq=2, B=2, T=64, H=2, dk=128, dv=128, dtype=1,
                chunk=64, ws=FAKE, ws_bytes=1 << 30, stream=None)
    args.update(over)
    return L.mdn_chunk_fwd_states(args["q"], args["k"], args["v"], args["alpha"],
                                  args["mu"], args["eta"], args["beta"], args["S0"],
                                  args["M0"], args["o"], args["S_T"], args["M_T"], Sc, Mc,
                                  args["cu"], args["n_seq"], args["B"], args["T"],
                                  args["H"], args["dk"], args["dv"], args["dtype"],
                                  args["chunk"], args["ws"], args["ws_bytes"],
                                  args["stream"])


SC, MC = ctypes.c_void_p(0x50000), ctypes.c_void_p(0x60000)


@pytest.mark.parametrize("Sc,Mc,over,code", [
    (None, MC, {}, 1),                               # both required when tokens exist
    (SC, None, {}, 1),
    (SC, SC, {}, 1),                                 # the same buffer twice
    (FAKE, MC, {}, 1),                               # aliases the inputs
    (ctypes.c_void_p(0x50008), MC, {}, 1),           # not 16-byte aligned
    (SC, MC, dict(S0=MC), 1),                        # aliases an initial state
    (SC, MC, dict(chunk=32), 2),                     # the rest as mdn_chunk_fwd
    (SC, MC, dict(q=None), 1),
])
def test_chunk_fwd_states_rejects(L, Sc, Mc, over, code):
    assert _chunk_states(L, Sc, Mc, **over) == code


def test_chunk_state_slots(L):
    # equal lengths: B * ceil(T / 64); packed: floor(T_total / 64) + n_seq
    assert mdn.chunk_state_slots(2, 2, 130, False) == 6
    assert mdn.chunk_state_slots(4, 4, 64, False) == 4
    assert mdn.chunk_state_slots(0, 0, 0, False) == 0
    assert mdn.chunk_state_slots(3, 1, 300, True) == 300 // 64 + 3
    assert mdn.chunk_state_slots(-1, 1, 10, False) == 0


def test_kernel_count_host_rules(L):
    # sequences under 128 chunks run as one pass on any device: prep + state
    # pass, plus the packed chunk offsets and the fp32 split of the inputs;
    # no tokens: one pass-through of the initial states; bad sizes: 0
    bf16, f32 = torch.bfloat16, torch.float32
    assert mdn.chunk_fwd_kernel_count(2, 2, 2048, 8, 128, bf16, False) == 2
    assert mdn.chunk_fwd_kernel_count(3, 1, 5000, 16, 128, bf16, True) == 3
    assert mdn.chunk_fwd_kernel_count(1, 1, 256, 2, 64, f32, False) == 3
    assert mdn.chunk_fwd_kernel_count(3, 1, 700, 4, 64, f32, True) == 4
    assert mdn.chunk_fwd_kernel_count(2, 2, 0, 4, 128, bf16, False) == 1
    assert mdn.chunk_fwd_kernel_count(1, 1, 64, 4, 96, bf16, False) == 0
    assert mdn.chunk_fwd_kernel_count(1, 1, 64, 0, 128, bf16, False) == 0
    assert mdn.chunk_fwd_kernel_count(0, 1, 64, 4, 128, bf16, False) == 0


def test_chunk_fwd_accepts_null_tensors_without_tokens(L):
    # no tokens: q, k, v, o and the gates may be null (empty tensors); the
    # call is not an argument error (it needs a device to go further)
    st = _chunk(L, q=None, k=None, v=None, o=None, alpha=None, mu=None, eta=None, T=0)
    assert st != mdn.MDN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library every call raises: there is no CPU or
    PyTorch fallback on the product path."""
    import subprocess
    import sys
    code = (
        "import momentum_delta_rule_gb300 as mdn\n"
        "mdn.LIB_PATH = %r\n"
        "try:\n"
        "    mdn.abi_version()\n"
        "except RuntimeError as e:\n"
        "    print('raised', 'not built' in str(e) or 'libmdn' in str(e))\n"
        "else:\n"
        "    print('returned')\n" % str(tmp_path / "absent" / "libmdn.so"))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "raised True", out.stdout + out.stderr


def _bwd(L, **over):
    P = lambda a: ctypes.c_void_p(a)
    args = dict(q=P(0x10000), k=P(0x11000), v=P(0x12000), alpha=P(0x13000), mu=P(0x14000),
                eta=P(0x15000), beta=None, Sc=P(0x16000), Mc=P(0x17000), do=P(0x18000),
                dS=None, dM=None, dq=P(0x20000), dk=P(0x21000), dv=P(0x22000),
                da=P(0x23000), dmu=P(0x24000), de=P(0x25000), db=None, dS0=None, dM0=None,
                cu=None, n_seq=2, B=2, T=64, H=2, dkd=128, dvd=128, dtype=1, chunk=64,
                ws=P(0x100000), ws_bytes=1 << 40, stream=None)
    args.update(over)
    a = args
    return L.mdn_chunk_bwd(a["q"], a["k"], a["v"], a["alpha"], a["mu"], a["eta"], a["beta"],
                           a["Sc"], a["Mc"], a.get("fws"), a["do"], a["dS"], a["dM"], a["dq"], a["dk"],
                           a["dv"], a["da"], a["dmu"], a["de"], a["db"], a["dS0"], a["dM0"],
                           a["cu"], a["n_seq"], a["B"], a["T"], a["H"], a["dkd"], a["dvd"],
                           a["dtype"], a["chunk"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(Sc=None), 1), (dict(do=None), 1), (dict(dq=None), 1), (dict(dmu=None), 1),
    (dict(dv=ctypes.c_void_p(0x10000)), 1),          # an output aliasing an input
    (dict(dk=ctypes.c_void_p(0x20000)), 1),          # two outputs the same
    (dict(dS0=ctypes.c_void_p(0x30008)), 1),         # misaligned
    (dict(fws=ctypes.c_void_p(0x200010)), 1),        # forward workspace not 256-aligned
    (dict(dq=ctypes.c_void_p(0x200000), fws=ctypes.c_void_p(0x200000)), 1),   # output aliasing it
    (dict(ws=None), 1), (dict(ws_bytes=256), 1),
    (dict(n_seq=3), 1), (dict(chunk=32), 2), (dict(dkd=96, dvd=96), 2),
])
def test_chunk_bwd_rejects(L, over, code):
    assert _bwd(L, **over) == code


def test_chunk_bwd_workspace_size(L):
    # per (chunk slot, head): the gradient block (five 64 x 64 fp32 matrices,
    # eight 64-float vector rows), then fp32 inputs: the fp32 chunk-end
    # adjoints and the residual adjoints; bf16 inputs: the adjoints as bf16
    # tiles and the tensor-core operand block (18 KiB)
    blk = 5 * 64 * 64 * 4 + 8 * 64 * 4
    slots = (16384 // 64 + 8) * 8
    meta = 2 * 256
    f32 = mdn.chunk_bwd_workspace_size(8, 16384, 8, 128, 0)
    bf16 = mdn.chunk_bwd_workspace_size(8, 16384, 8, 128, 1)
    assert f32 == meta + slots * (blk + 2 * 128 * 128 * 4 + 64 * 128 * 4)
    assert bf16 == meta + slots * (blk + 2 * 128 * 128 * 2 + 18432)
    assert f32 % 256 == 0 and bf16 % 256 == 0
    assert mdn.chunk_bwd_workspace_size(-1, 10, 1, 64, 1) == 0


def _block(L, **over):
    P = lambda a: ctypes.c_void_p(a)
    args = dict(x=P(0x10000), W_in=P(0x20000), conv=P(0x30000), rms=P(0x40000), W_o=P(0x50000),
                a=1.0, b=0.0, s=1.0, tau=1.0, lmin=-2.0, cd=0.0, eps=1e-6, S0=None, M0=None,
                y=P(0x60000), S_T=None, M_T=None, cu=None, n_seq=2, B=2, T=64, H=2, d=128,
                dm=256, dtype=1, ws=P(0x100000), ws_bytes=1 << 40, stream=None)
    args.update(over)
    a = args
    return L.mdn_block_fwd(a["x"], a["W_in"], a["conv"], a["rms"], a["W_o"], a["a"], a["b"],
                           a["s"], a["tau"], a["lmin"], a["cd"], a["eps"], a["S0"], a["M0"],
                           a["y"], a["S_T"], a["M_T"], a["cu"], a["n_seq"], a["B"], a["T"],
                           a["H"], a["d"], a["dm"], a["dtype"], a["ws"], a["ws_bytes"],
                           a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(x=None), 1), (dict(W_o=None), 1), (dict(conv=None), 1),
    (dict(y=ctypes.c_void_p(0x60008)), 1), (dict(ws=None), 1), (dict(ws_bytes=1024), 1),
    (dict(n_seq=3), 1), (dict(dtype=4), 1), (dict(eps=-1.0), 1),
    (dict(d=96), 2), (dict(dm=100), 2),
])
def test_block_fwd_rejects(L, over, code):
    assert _block(L, **over) == code
