"""The kernels' bounded pipeline waits, run out on purpose.

Every mbarrier wait in the prefill and backward kernels gives up after
GQA_WAIT_TIMEOUT_NS: the CTA raises GQA_ERR_DEVICE_TIMEOUT, drains the copies
and matrix products it has in flight, frees its tensor memory and exits --
no trap, so the CUDA context stays usable.  With GQA_TEST_FORCE_TIMEOUT set,
one MMA-issuing thread per CTA first waits on a barrier that nothing arrives
on, so the wait certainly runs out (after a 20 us limit here) and every other
role of the CTA has to notice the abort in its own waits.

The checks run in a child process (both variables are read at each call, so
one process can set and clear them):
  1. each entry point with such waits -- dense prefill at D = 64 and 128,
     packed and block-sparse prefill, the backward -- returns, and
     gqa_device_status() reports GQA_ERR_DEVICE_TIMEOUT (then OK once read);
  2. with a 1 ns limit and no forced stall, waits give up wherever they
     happen to poll: every call still returns, with either status;
  3. with the variables cleared, the same calls in the same process match the
     oracle, and 130 more prefill launches (every work-unit scheduler slot
     reused twice after the aborted launches) give bitwise the first result.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.gpu
def test_wait_timeouts_abort_cleanly_and_the_context_stays_usable():
    env = dict(os.environ)
    env.pop("GQA_WAIT_TIMEOUT_NS", None)
    env.pop("GQA_TEST_FORCE_TIMEOUT", None)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--child"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, "child failed:\n%s\n%s" % (r.stdout[-3000:], r.stderr[-3000:])
    assert "CHILD OK" in r.stdout, r.stdout[-3000:]


def _child():
    sys.path.insert(0, ROOT)
    sys.path.insert(0, HERE)
    import time

    import numpy as np
    import torch

    import grouped_query_attention_08_b300 as gqa
    import oracle
    from grouped_query_attention_08_b300 import build, inputs
    from parity import compare, to_dev

    build.build()
    gqa.load_library()
    torch.cuda.set_device(0)

    pre64 = inputs.make_prefill(2, 12, 3, 700, 700, 64, seed=31, lens=(300, 700), dtype="bf16")
    pre128 = inputs.make_prefill(1, 16, 4, 600, 600, 128, seed=32, dtype="bf16")
    var = inputs.make_varlen(3, 8, 2, 64, seed=33, lens=[300, 17, 420], dtype="bf16")
    sp = inputs.make_prefill(1, 8, 2, 500, 500, 64, seed=34, dtype="bf16")
    bm = inputs.make_block_mask(4, 4, "random", density=0.6, seed=34)
    bwd = inputs.make_backward(2, 8, 2, 400, 400, 64, seed=35, lens=(200, 400))
    d64, d128, dv, ds, db = to_dev(pre64), to_dev(pre128), to_dev(var), to_dev(sp), to_dev(bwd)
    bmd = bm.cuda()
    out_b, lse_b = gqa.gqa_fwd(db["q"], db["k"], db["v"], seqlens_k=db["seqlens_k"], scale=0.125)
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0

    calls = {
        "prefill D64": lambda: gqa.gqa_fwd(d64["q"], d64["k"], d64["v"], seqlens_k=d64["seqlens_k"], scale=0.125),
        "prefill D128 causal": lambda: gqa.gqa_fwd(d128["q"], d128["k"], d128["v"], causal=True, scale=0.088),
        "varlen": lambda: gqa.gqa_fwd_varlen(dv["q"], dv["k"], dv["v"], dv["cu_seqlens_q"], dv["cu_seqlens_k"],
                                             max_seqlen_q=dv["max_seqlen_q"], max_seqlen_k=dv["max_seqlen_k"],
                                             scale=0.125),
        "sparse": lambda: gqa.gqa_fwd_sparse(ds["q"], ds["k"], ds["v"], bmd, 128, scale=0.125),
        "backward": lambda: gqa.gqa_bwd(db["q"], db["k"], db["v"], out_b, db["dout"], lse_b,
                                        seqlens_k=db["seqlens_k"], scale=0.125),
    }

    # 1. forced: one wait per CTA cannot complete and runs out after 20 us
    os.environ["GQA_WAIT_TIMEOUT_NS"] = "20000"
    os.environ["GQA_TEST_FORCE_TIMEOUT"] = "1"
    for name, fn in calls.items():
        t0 = time.perf_counter()
        fn()
        st = gqa.gqa_device_status()          # synchronises: the kernels have returned
        dt = time.perf_counter() - t0
        assert st == gqa.GQA_ERR_DEVICE_TIMEOUT, (name, gqa.gqa_status_string(st))
        assert gqa.gqa_device_status() == 0, name          # cleared by the read
        print("forced timeout: %-20s status %s, %.1f ms" % (name, gqa.gqa_status_string(st), dt * 1e3))

    # 2. a 1 ns limit: waits give up wherever they happen to poll
    del os.environ["GQA_TEST_FORCE_TIMEOUT"]
    os.environ["GQA_WAIT_TIMEOUT_NS"] = "1"
    for rep in range(3):
        for name, fn in calls.items():
            fn()
            st = gqa.gqa_device_status()
            assert st in (gqa.GQA_OK, gqa.GQA_ERR_DEVICE_TIMEOUT), (name, st)
            print("1 ns limit: %-20s status %s" % (name, gqa.gqa_status_string(st)))

    # 3. default limit again, same process: results match the oracle
    del os.environ["GQA_WAIT_TIMEOUT_NS"]
    out, lse = calls["prefill D64"]()
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    ref, _ = oracle.attention(pre64["q"], pre64["k"], pre64["v"], scale=0.125, seqlens_k=pre64["seqlens_k"])
    compare(out.float().cpu().numpy(), ref, torch.bfloat16, what="prefill D64 after the timeouts")
    o128, _ = calls["prefill D128 causal"]()
    ref128, _ = oracle.attention(pre128["q"], pre128["k"], pre128["v"], scale=0.088, causal=True)
    compare(o128.float().cpu().numpy(), ref128, torch.bfloat16, what="prefill D128 after the timeouts")
    ov, _ = calls["varlen"]()
    refv, _ = oracle.attention_varlen(var["q"], var["k"], var["v"], var["cu_seqlens_q"], var["cu_seqlens_k"],
                                      scale=0.125)
    compare(ov.float().cpu().numpy(), refv, torch.bfloat16, what="varlen after the timeouts")
    osp, _ = calls["sparse"]()
    refs, _ = oracle.attention_blockmask(sp["q"], sp["k"], sp["v"], bm, 128, scale=0.125)
    compare(osp.float().cpu().numpy(), refs, torch.bfloat16, what="sparse after the timeouts")
    gq, gk, gv = calls["backward"]()
    rq, rk, rv = oracle.attention_backward(bwd["q"], bwd["k"], bwd["v"], bwd["dout"], scale=0.125,
                                           seqlens_k=bwd["seqlens_k"])
    for got, r, what in ((gq, rq, "dq"), (gk, rk, "dk"), (gv, rv, "dv")):
        e = np.abs(got.float().cpu().numpy() - r)
        assert e.max() <= 2e-2 * np.abs(r).max() + 1e-4, (what, float(e.max()))
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0

    # every scheduler slot reused twice after the aborted launches
    first = out.clone()
    for _ in range(130):
        out, _ = calls["prefill D64"]()
    torch.cuda.synchronize()
    assert gqa.gqa_device_status() == 0
    assert torch.equal(out, first)
    print("CHILD OK")


if __name__ == "__main__" and "--child" in sys.argv:
    _child()
