"""Host-side tests of the C ABI (no GPU needed): the library loads, exports every
function declared in include/palimpsa.h, and rejects bad arguments with status
codes before touching a device."""
import ctypes
import os
import re

import pytest

import metaplastic_linear_attention_gb300 as pal
from metaplastic_linear_attention_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "palimpsa.h")

(OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_DOMAIN, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT,
 ERR_SCRATCH_LIMIT) = range(10)


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return pal.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(palimpsa_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("palimpsa_forward_chunked", "palimpsa_step", "palimpsa_status_string",
                     "palimpsa_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in palimpsa.h but not exported"


def test_abi_version_and_status_strings(lib):
    assert pal.palimpsa_abi_version() == 1
    seen = set()
    for code in range(10):
        s = pal.palimpsa_status_string(code)
        assert s and s not in seen
        seen.add(s)
    assert pal.palimpsa_status_string(99) == "unknown status"


# Fake, well-aligned addresses: every check below fails before any pointer is used.
P = 1 << 20


def _fwd(lib, **over):
    args = dict(q=P, k=P, v=P, beta=P, d_t=P, A=P, I_prior=P, mu0=None, I0=None, y=P, mu_T=P, I_T=P,
                B=1, H=2, T=16, d_k=128, d_v=64, chunk=0, dtype=1)
    args.update(over)
    return lib.palimpsa_forward_chunked(
        args["q"], args["k"], args["v"], args["beta"], args["d_t"], args["A"], args["I_prior"], args["mu0"],
        args["I0"], args["y"], args["mu_T"], args["I_T"], args["B"], args["H"], args["T"], args["d_k"],
        args["d_v"], args["chunk"], args["dtype"], None)


def _step(lib, **over):
    args = dict(q=P, k=P, v=P, beta=P, d_t=P, A=P, I_prior=P, mu=P, I=P, y=P, B=4, H=2, d_k=128, d_v=64,
                dtype=1)
    args.update(over)
    return lib.palimpsa_step(args["q"], args["k"], args["v"], args["beta"], args["d_t"], args["A"],
                             args["I_prior"], args["mu"], args["I"], args["y"], args["B"], args["H"],
                             args["d_k"], args["d_v"], args["dtype"], None)


@pytest.mark.parametrize("field", ["q", "k", "v", "beta", "d_t", "A", "I_prior", "y", "mu_T", "I_T"])
def test_forward_rejects_null(lib, field):
    assert _fwd(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("field", ["A", "I_prior", "mu_T", "I_T"])
def test_forward_empty_sequence_still_needs_state_and_gates(lib, field):
    assert _fwd(lib, T=0, q=None, k=None, v=None, beta=None, d_t=None, y=None, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("field", ["q", "k", "v", "beta", "d_t", "A", "I_prior", "mu", "I", "y"])
def test_step_rejects_null(lib, field):
    assert _step(lib, **{field: None}) == ERR_NULL


@pytest.mark.parametrize("over,code", [
    (dict(dtype=2), ERR_DTYPE), (dict(dtype=-1), ERR_DTYPE),
    (dict(B=0), ERR_SHAPE), (dict(H=0), ERR_SHAPE), (dict(T=-1), ERR_SHAPE), (dict(B=-3), ERR_SHAPE),
    (dict(d_k=96), ERR_UNSUPPORTED), (dict(d_k=32), ERR_UNSUPPORTED), (dict(d_v=12), ERR_UNSUPPORTED),
    (dict(d_v=0), ERR_UNSUPPORTED), (dict(d_v=264), ERR_UNSUPPORTED), (dict(chunk=48), ERR_UNSUPPORTED),
    (dict(chunk=256), ERR_UNSUPPORTED), (dict(chunk=8), ERR_UNSUPPORTED),
    (dict(q=P + 8), ERR_ALIGN), (dict(v=P + 4), ERR_ALIGN), (dict(y=P + 2), ERR_ALIGN),
    (dict(mu0=P + 8), ERR_ALIGN), (dict(I0=P + 4), ERR_ALIGN), (dict(d_t=P + 2), ERR_ALIGN),
])
def test_forward_rejects_bad_arguments(lib, over, code):
    assert _fwd(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(dtype=7), ERR_DTYPE), (dict(B=0), ERR_SHAPE), (dict(H=-1), ERR_SHAPE),
    (dict(d_k=256), ERR_UNSUPPORTED), (dict(d_v=7), ERR_UNSUPPORTED),
    (dict(mu=P + 8), ERR_ALIGN), (dict(k=P + 2), ERR_ALIGN), (dict(A=P + 1), ERR_ALIGN),
])
def test_step_rejects_bad_arguments(lib, over, code):
    assert _step(lib, **over) == code


def test_binding_raises_without_fallback(tmp_path):
    """A missing library is an error, never a silent CPU path."""
    import metaplastic_linear_attention_gb300.binding as b
    saved = b._lib
    try:
        b._lib = None
        with pytest.raises(RuntimeError):
            b.load_library(str(tmp_path / "libpalimpsa.so"))
    finally:
        b._lib = saved


def test_product_path_does_not_import_the_oracle():
    """The package never imports the oracle (the oracle is test infrastructure)."""
    pkg = os.path.join(ROOT, "metaplastic_linear_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "palimpsa_oracle" not in text, f


@pytest.mark.parametrize("entry", ["palimpsa_forward_chunked", "palimpsa_forward_chunked_noalloc"])
@pytest.mark.parametrize("over,code", [
    (dict(q=None), ERR_NULL), (dict(I_T=None), ERR_NULL), (dict(dtype=3), ERR_DTYPE), (dict(H=0), ERR_SHAPE),
    (dict(d_k=96), ERR_UNSUPPORTED), (dict(mu_T=P + 4), ERR_ALIGN),
])
def test_both_forward_entry_points_validate_alike(lib, entry, over, code):
    args = dict(q=P, k=P, v=P, beta=P, d_t=P, A=P, I_prior=P, mu0=None, I0=None, y=P, mu_T=P, I_T=P,
                B=1, H=2, T=16, d_k=128, d_v=64, chunk=0, dtype=1)
    args.update(over)
    fn = getattr(lib, entry)
    assert fn(args["q"], args["k"], args["v"], args["beta"], args["d_t"], args["A"], args["I_prior"], args["mu0"],
              args["I0"], args["y"], args["mu_T"], args["I_T"], args["B"], args["H"], args["T"], args["d_k"],
              args["d_v"], args["chunk"], args["dtype"], None) == code


def _fused(lib, **over):
    args = dict(q=P, k=P, v=P, b=P, d=P, A=P, I_prior=P, b_scale=None, mu0=None, I0=None, y=P, mu_T=P, I_T=P,
                B=1, H=2, T=16, d_k=128, d_v=64, chunk=0, flags=3, dtype=1)
    args.update(over)
    return lib.palimpsa_forward_fused(
        args["q"], args["k"], args["v"], args["b"], args["d"], args["A"], args["I_prior"], args["b_scale"],
        args["mu0"], args["I0"], args["y"], args["mu_T"], args["I_T"], args["B"], args["H"], args["T"],
        args["d_k"], args["d_v"], args["chunk"], args["flags"], args["dtype"], None)


def _step_fused(lib, **over):
    args = dict(q=P, k=P, v=P, b=P, d=P, A=P, I_prior=P, b_scale=None, mu=P, I=P, y=P, B=4, H=2, d_k=128, d_v=64,
                flags=1, dtype=1)
    args.update(over)
    return lib.palimpsa_step_fused(args["q"], args["k"], args["v"], args["b"], args["d"], args["A"],
                                   args["I_prior"], args["b_scale"], args["mu"], args["I"], args["y"], args["B"],
                                   args["H"], args["d_k"], args["d_v"], args["flags"], args["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(flags=4), ERR_UNSUPPORTED), (dict(flags=0x80000000), ERR_UNSUPPORTED),
    (dict(b_scale=P + 2), ERR_ALIGN), (dict(q=None), ERR_NULL), (dict(d=None), ERR_NULL),
    (dict(I_T=None), ERR_NULL), (dict(dtype=5), ERR_DTYPE), (dict(T=-1), ERR_SHAPE),
    (dict(d_k=96), ERR_UNSUPPORTED), (dict(chunk=24), ERR_UNSUPPORTED), (dict(v=P + 8), ERR_ALIGN),
    (dict(d=P + 1), ERR_ALIGN),
])
def test_forward_fused_rejects_bad_arguments(lib, over, code):
    assert _fused(lib, **over) == code


@pytest.mark.parametrize("over,code", [
    (dict(flags=8), ERR_UNSUPPORTED), (dict(b_scale=P + 1), ERR_ALIGN), (dict(b=None), ERR_NULL),
    (dict(mu=None), ERR_NULL), (dict(dtype=-2), ERR_DTYPE), (dict(B=0), ERR_SHAPE), (dict(d_v=20), ERR_UNSUPPORTED),
    (dict(I=P + 4), ERR_ALIGN),
])
def test_step_fused_rejects_bad_arguments(lib, over, code):
    assert _step_fused(lib, **over) == code


def _varlen(lib, **over):
    args = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, mu0=None, I0=None, y=P, mu_T=P, I_T=P, cu=P, N=3, H=2,
                total_T=100, max_seqlen=50, d_k=128, d_v=64, chunk=0, dtype=1)
    args.update(over)
    return lib.palimpsa_forward_varlen(
        args["q"], args["k"], args["v"], args["beta"], args["d"], args["A"], args["I_prior"], args["mu0"],
        args["I0"], args["y"], args["mu_T"], args["I_T"], args["cu"], args["N"], args["H"], args["total_T"],
        args["max_seqlen"], args["d_k"], args["d_v"], args["chunk"], args["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(cu=None), ERR_NULL), (dict(q=None), ERR_NULL), (dict(mu_T=None), ERR_NULL),
    (dict(cu=P + 2), ERR_ALIGN), (dict(y=P + 8), ERR_ALIGN), (dict(N=0), ERR_SHAPE), (dict(H=0), ERR_SHAPE),
    (dict(total_T=-1), ERR_SHAPE), (dict(max_seqlen=-1), ERR_SHAPE), (dict(max_seqlen=101), ERR_SHAPE),
    (dict(dtype=9), ERR_DTYPE), (dict(d_v=4), ERR_UNSUPPORTED), (dict(chunk=8), ERR_UNSUPPORTED),
])
def test_forward_varlen_rejects_bad_arguments(lib, over, code):
    assert _varlen(lib, **over) == code


def test_forward_varlen_empty_tokens_need_no_token_arrays(lib):
    # total_T = 0: every sequence is empty; the token arrays are not read and may be
    # NULL, but the state arrays and offsets are still required
    assert _varlen(lib, total_T=0, max_seqlen=0, q=None, k=None, v=None, beta=None, d=None, y=None,
                   mu_T=None) == ERR_NULL


@pytest.mark.parametrize("over,code", [
    (dict(summary=None), ERR_NULL), (dict(gamma=None), ERR_NULL), (dict(q=None), ERR_NULL),
    (dict(summary=P + 4), ERR_ALIGN), (dict(gamma=P + 2), ERR_ALIGN), (dict(T=-2), ERR_SHAPE),
    (dict(d_k=32), ERR_UNSUPPORTED), (dict(dtype=3), ERR_DTYPE),
])
def test_segment_summary_rejects_bad_arguments(lib, over, code):
    args = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, summary=P, gamma=P, B=1, H=2, T=16, d_k=128, d_v=64,
                chunk=0, dtype=1)
    args.update(over)
    assert lib.palimpsa_segment_summary(args["q"], args["k"], args["v"], args["beta"], args["d"], args["A"],
                                        args["I_prior"], args["summary"], args["gamma"], args["B"], args["H"],
                                        args["T"], args["d_k"], args["d_v"], args["chunk"], args["dtype"],
                                        None) == code


@pytest.mark.parametrize("over,code", [
    (dict(S=None), ERR_NULL), (dict(G=None), ERR_NULL), (dict(I_prior=None), ERR_NULL), (dict(mu=None), ERR_NULL),
    (dict(R=-1), ERR_SHAPE), (dict(B=0), ERR_SHAPE), (dict(S=P + 8), ERR_ALIGN), (dict(I=P + 4), ERR_ALIGN),
    (dict(G=P + 1), ERR_ALIGN), (dict(d_v=12), ERR_UNSUPPORTED),
])
def test_state_combine_rejects_bad_arguments(lib, over, code):
    args = dict(S=P, G=P, R=3, I_prior=P, mu0=None, I0=None, mu=P, I=P, B=1, H=2, d_k=128, d_v=64)
    args.update(over)
    assert lib.palimpsa_state_combine(args["S"], args["G"], args["R"], args["I_prior"], args["mu0"], args["I0"],
                                      args["mu"], args["I"], args["B"], args["H"], args["d_k"], args["d_v"],
                                      None) == code


@pytest.mark.parametrize("over,code", [
    (dict(segments=None), ERR_NULL), (dict(scratch=None), ERR_NULL), (dict(dtype=4), ERR_DTYPE),
    (dict(B=0), ERR_SHAPE), (dict(T=-1), ERR_SHAPE), (dict(d_k=96), ERR_UNSUPPORTED), (dict(chunk=48), ERR_UNSUPPORTED),
])
def test_forward_plan_rejects_bad_arguments(lib, over, code):
    seg, sl, ln, sb = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    args = dict(B=4, H=16, T=2048, d_k=128, d_v=64, chunk=0, dtype=1, segments=ctypes.byref(seg),
                seg_len=ctypes.byref(sl), launches=ctypes.byref(ln), scratch=ctypes.byref(sb))
    args.update(over)
    assert lib.palimpsa_forward_plan(args["B"], args["H"], args["T"], args["d_k"], args["d_v"], args["chunk"],
                                     args["dtype"], args["segments"], args["seg_len"], args["launches"],
                                     args["scratch"]) == code


def test_checkpoint_bytes_formula(lib):
    lib.palimpsa_checkpoint_bytes.restype = ctypes.c_size_t
    assert lib.palimpsa_checkpoint_bytes(4, 16, 2048, 128, 64) == 4 * 16 * 64 * 64 * 2 * 128 * 4
    assert lib.palimpsa_checkpoint_bytes(1, 2, 33, 64, 8) == 1 * 2 * 2 * 8 * 2 * 64 * 4
    assert lib.palimpsa_checkpoint_bytes(1, 1, 0, 128, 64) == 0
    assert lib.palimpsa_checkpoint_bytes(0, 1, 10, 128, 64) == 0


@pytest.mark.parametrize("over,code", [(dict(ck=None), ERR_NULL), (dict(ck=P + 4), ERR_ALIGN),
                                       (dict(q=None), ERR_NULL), (dict(d_k=96), ERR_UNSUPPORTED)])
def test_forward_checkpointed_rejects_bad_arguments(lib, over, code):
    args = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, mu0=None, I0=None, y=P, mu_T=P, I_T=P, ck=P, B=1, H=2,
                T=16, d_k=128, d_v=64, chunk=0, dtype=1)
    args.update(over)
    assert lib.palimpsa_forward_checkpointed(
        args["q"], args["k"], args["v"], args["beta"], args["d"], args["A"], args["I_prior"], args["mu0"], args["I0"],
        args["y"], args["mu_T"], args["I_T"], args["ck"], args["B"], args["H"], args["T"], args["d_k"], args["d_v"],
        args["chunk"], args["dtype"], None) == code


@pytest.mark.parametrize("over,code", [(dict(ck=None), ERR_NULL), (dict(ck=P + 8), ERR_ALIGN),
                                       (dict(dy=None), ERR_NULL), (dict(dtype=7), ERR_DTYPE)])
def test_backward_checkpointed_rejects_bad_arguments(lib, over, code):
    a = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, mu0=None, I0=None, dy=P, dmu=None, dI=None, dq=P, dk=P, dv=P,
             db=P, dd=P, dA=P, dIp=P, dmu0=None, dI0=None, ck=P, B=1, H=2, T=16, d_k=128, d_v=64, dtype=1)
    a.update(over)
    assert lib.palimpsa_backward_checkpointed(
        a["q"], a["k"], a["v"], a["beta"], a["d"], a["A"], a["I_prior"], a["mu0"], a["I0"], a["dy"], a["dmu"], a["dI"],
        a["dq"], a["dk"], a["dv"], a["db"], a["dd"], a["dA"], a["dIp"], a["dmu0"], a["dI0"], a["ck"], a["B"], a["H"],
        a["T"], a["d_k"], a["d_v"], a["dtype"], None) == code


def _seq(lib, **over):
    args = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, mu=P, I=P, y=P, S=4, B=4, H=2, d_k=128, d_v=64, dtype=1)
    args.update(over)
    return lib.palimpsa_step_sequence(args["q"], args["k"], args["v"], args["beta"], args["d"], args["A"],
                                      args["I_prior"], args["mu"], args["I"], args["y"], args["S"], args["B"],
                                      args["H"], args["d_k"], args["d_v"], args["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(S=-1), ERR_SHAPE), (dict(q=None), ERR_NULL), (dict(mu=None), ERR_NULL), (dict(dtype=3), ERR_DTYPE),
    (dict(B=0), ERR_SHAPE), (dict(d_v=12), ERR_UNSUPPORTED), (dict(y=P + 4), ERR_ALIGN),
])
def test_step_sequence_rejects_bad_arguments(lib, over, code):
    assert _seq(lib, **over) == code


def test_step_sequence_of_no_tokens_does_nothing(lib):
    # S = 0 returns before any pointer is looked at or any device call is made
    assert _seq(lib, S=0, q=None, k=None, v=None, beta=None, d=None, y=None) == OK


@pytest.mark.parametrize("over,code", [(dict(flags=8), ERR_UNSUPPORTED), (dict(b_scale=P + 2), ERR_ALIGN),
                                       (dict(cu=None), ERR_NULL), (dict(max_seqlen=200), ERR_SHAPE)])
def test_forward_varlen_fused_rejects_bad_arguments(lib, over, code):
    a = dict(q=P, k=P, v=P, b=P, d=P, A=P, I_prior=P, b_scale=None, mu0=None, I0=None, y=P, mu_T=P, I_T=P, cu=P, N=3,
             H=2, total_T=100, max_seqlen=50, d_k=128, d_v=64, chunk=0, flags=1, dtype=1)
    a.update(over)
    assert lib.palimpsa_forward_varlen_fused(
        a["q"], a["k"], a["v"], a["b"], a["d"], a["A"], a["I_prior"], a["b_scale"], a["mu0"], a["I0"], a["y"],
        a["mu_T"], a["I_T"], a["cu"], a["N"], a["H"], a["total_T"], a["max_seqlen"], a["d_k"], a["d_v"], a["chunk"],
        a["flags"], a["dtype"], None) == code


def _bwd_varlen(lib, **over):
    a = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, mu0=None, I0=None, dy=P, dmu=None, dI=None, dq=P, dk=P, dv=P,
             db=P, dd=P, dA=P, dIp=P, dmu0=None, dI0=None, ck=None, cu=P, N=3, H=2, total_T=100, max_seqlen=50,
             d_k=128, d_v=64, dtype=1)
    a.update(over)
    return lib.palimpsa_backward_varlen(
        a["q"], a["k"], a["v"], a["beta"], a["d"], a["A"], a["I_prior"], a["mu0"], a["I0"], a["dy"], a["dmu"], a["dI"],
        a["dq"], a["dk"], a["dv"], a["db"], a["dd"], a["dA"], a["dIp"], a["dmu0"], a["dI0"], a["ck"], a["cu"], a["N"],
        a["H"], a["total_T"], a["max_seqlen"], a["d_k"], a["d_v"], a["dtype"], None)


@pytest.mark.parametrize("over,code", [
    (dict(cu=None), ERR_NULL), (dict(dy=None), ERR_NULL), (dict(dA=None), ERR_NULL), (dict(cu=P + 2), ERR_ALIGN),
    (dict(ck=P + 4), ERR_ALIGN), (dict(dq=P + 8), ERR_ALIGN), (dict(N=0), ERR_SHAPE), (dict(total_T=-1), ERR_SHAPE),
    (dict(max_seqlen=101), ERR_SHAPE), (dict(max_seqlen=-1), ERR_SHAPE), (dict(dtype=4), ERR_DTYPE),
    (dict(d_k=32), ERR_UNSUPPORTED),
])
def test_backward_varlen_rejects_bad_arguments(lib, over, code):
    assert _bwd_varlen(lib, **over) == code


def test_backward_varlen_empty_tokens_need_no_token_arrays(lib):
    # total_T = 0: the token arrays may be NULL; the per-head gradients may not
    assert _bwd_varlen(lib, total_T=0, max_seqlen=0, q=None, k=None, v=None, beta=None, d=None, dy=None, dq=None,
                       dk=None, dv=None, db=None, dd=None, dA=None) == ERR_NULL


@pytest.mark.parametrize("over,code", [(dict(ck=None), ERR_NULL), (dict(ck=P + 4), ERR_ALIGN),
                                       (dict(cu=None), ERR_NULL), (dict(max_seqlen=101), ERR_SHAPE)])
def test_forward_varlen_checkpointed_rejects_bad_arguments(lib, over, code):
    a = dict(q=P, k=P, v=P, beta=P, d=P, A=P, I_prior=P, mu0=None, I0=None, y=P, mu_T=P, I_T=P, ck=P, cu=P, N=3, H=2,
             total_T=100, max_seqlen=50, d_k=128, d_v=64, chunk=0, dtype=1)
    a.update(over)
    assert lib.palimpsa_forward_varlen_checkpointed(
        a["q"], a["k"], a["v"], a["beta"], a["d"], a["A"], a["I_prior"], a["mu0"], a["I0"], a["y"], a["mu_T"],
        a["I_T"], a["ck"], a["cu"], a["N"], a["H"], a["total_T"], a["max_seqlen"], a["d_k"], a["d_v"], a["chunk"],
        a["dtype"], None) == code


def test_checkpoint_bytes_varlen_formula(lib):
    # per head total_T // 32 + N slots of d_v x 2 x d_k floats: proportional to the
    # tokens, whatever the longest sequence
    lib.palimpsa_checkpoint_bytes_varlen.restype = ctypes.c_size_t
    assert lib.palimpsa_checkpoint_bytes_varlen(5, 16, 2048, 128, 64) == 16 * (64 + 5) * 64 * 2 * 128 * 4
    assert lib.palimpsa_checkpoint_bytes_varlen(3, 2, 31, 64, 8) == 2 * (0 + 3) * 8 * 2 * 64 * 4
    assert lib.palimpsa_checkpoint_bytes_varlen(0, 2, 31, 64, 8) == 0
    assert lib.palimpsa_checkpoint_bytes_varlen(2, 1, -1, 128, 64) == 0


def test_packed_checkpoint_slots_never_overlap():
    """The slot rule for packed checkpoints (sequence n from token s0 owns slots
    s0 // 32 + n onwards, ceil(L / 32) of them): no two sequences share a slot and
    every slot lies inside total_T // 32 + N, over many random length mixes."""
    import random
    rnd = random.Random(5)
    for _ in range(2000):
        N = rnd.randint(1, 12)
        lengths = [rnd.choice([0, 1, 31, 32, 33, 63, 64, 65, rnd.randint(0, 300)]) for _ in range(N)]
        gap = rnd.randint(0, 40)
        total = sum(lengths) + gap
        used = set()
        s0 = 0
        for n, L in enumerate(lengths):
            slots = {s0 // 32 + n + c for c in range(-(-L // 32))}
            assert not (slots & used) and all(0 <= x < total // 32 + N for x in slots), (lengths, n)
            used |= slots
            s0 += L


@pytest.mark.parametrize("over,code", [(dict(S=-1), ERR_SHAPE), (dict(flags=16), ERR_UNSUPPORTED),
                                       (dict(q=None), ERR_NULL), (dict(b_scale=P + 2), ERR_ALIGN)])
def test_step_sequence_fused_rejects_bad_arguments(lib, over, code):
    a = dict(q=P, k=P, v=P, b=P, d=P, A=P, I_prior=P, b_scale=None, mu=P, I=P, y=P, S=4, B=4, H=2, d_k=128, d_v=64,
             flags=1, dtype=1)
    a.update(over)
    assert lib.palimpsa_step_sequence_fused(
        a["q"], a["k"], a["v"], a["b"], a["d"], a["A"], a["I_prior"], a["b_scale"], a["mu"], a["I"], a["y"], a["S"],
        a["B"], a["H"], a["d_k"], a["d_v"], a["flags"], a["dtype"], None) == code


def test_packed_checkpoint_shape_matches_the_library_size(lib):
    # the binding allocates packed checkpoints from packed_checkpoint_shape; the
    # library sizes them with palimpsa_checkpoint_bytes_varlen: the two must agree
    import math
    for N, H, total_T, d_k, d_v in ((1, 1, 0, 64, 8), (5, 16, 2048, 128, 64), (7, 3, 1001, 64, 40),
                                    (64, 32, 131072, 128, 64)):
        shape = pal.packed_checkpoint_shape(N, H, total_T, d_k, d_v)
        assert math.prod(shape) * 4 == pal.palimpsa_checkpoint_bytes_varlen(N, H, total_T, d_k, d_v)


def test_scratch_query_rejects_null(lib):
    assert lib.palimpsa_scratch_reserved_bytes(None) == ERR_NULL


def test_issue_rate_probe_rejects_bad_arguments(lib):
    import ctypes
    out = ctypes.c_double()
    assert lib.palimpsa_probe_issue_rate(0, None, None) == ERR_NULL
    assert lib.palimpsa_probe_issue_rate(-1, ctypes.byref(out), None) == ERR_UNSUPPORTED
    assert lib.palimpsa_probe_issue_rate(5, ctypes.byref(out), None) == ERR_UNSUPPORTED
    assert set(pal.binding.PROBE_OPS) == {"rcp", "ex2", "ffma", "rsqrt", "lg2"}
