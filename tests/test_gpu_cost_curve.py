"""The online verify-cost curve on the GPU: P3 "Teaching the Speculator What a Draft Costs",
"What we changed" (event pairs around real verify steps, read without waiting) and "The
controller, and the table it reads from" (the controller reads the rebuilt table).

* Real verify steps of two batch sizes are filed under their token counts; their medians
  replace the boot values there and nowhere else.
* A token count held on the device (adaptive_pick_k's cu_drafts_out[B] plus B bonus rows) is
  read back after the step and the observation lands at that count.
* poll() never waits: a step still running on the stream stays pending.
* upload() changes what the adaptive pipeline's graph picks at its next launch.
* begin() on a stream being captured is refused.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_block_verify_gb300 as sv  # noqa: E402
from speculative_decoding_block_verify_gb300 import workloads  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sv.lib()


def _verify_inputs(B, seed):
    inp = workloads.make_verify_inputs("batch64", seed, B=B, N=5, V=32768)
    return inp, parity.verify_to_device(inp, torch)


def test_real_verify_steps_are_filed_under_their_token_counts():
    boot = np.full(129, 1000.0, np.float32)
    c = sv.CostCurve(boot, window=32, min_samples=3, rebuild_every=32)
    counts = {}
    for B, seed in ((4, 11), (16, 12)):
        inp, d = _verify_inputs(B, seed)
        n_tok = int(inp["cu_drafts"][-1]) + B
        counts[n_tok] = 0
        for step in range(20):
            c.begin()
            sv.spec_verify_block(d["cu"], d["dq"], d["dp"], d["x"], d["T"], 5, 0, step)
            c.end(n_tok)
            counts[n_tok] += 1
            c.poll()
    torch.cuda.synchronize()
    c.poll()
    t, cnt = c.table()
    assert cnt["observations"] == 40 and cnt["pending"] == 0 and cnt["dropped"] == 0
    assert cnt["rebuilds"] == 1
    for n, v in enumerate(t):
        if n in counts:
            assert 0.0 < v < 50.0, (n, v)   # a verify of at most 96 rows of 32768: well under 50 ms
        else:
            assert v == 1000.0
    c.close()


def test_device_token_count_is_read_after_the_step():
    B, kmax, H = 8, 5, 256
    conf = workloads.make_confidence_inputs(3, B=B, kmax=kmax, H=H, n_max=64)
    hidden = torch.as_tensor(np.asarray(conf["hidden"], np.float32)).cuda().to(torch.bfloat16)
    w = torch.as_tensor(np.asarray(conf["w"], np.float32)).cuda().to(torch.bfloat16)
    vm = torch.as_tensor((2.0 + 0.4 * np.arange(65)).astype(np.float32)).cuda()
    c = sv.CostCurve(np.full(65, 7.0, np.float32), window=4, min_samples=1, rebuild_every=1)
    pk = None
    for _ in range(3):
        c.begin()
        pk = sv.adaptive_pick_k(hidden, w, 0.0, vm)
        c.end(B, device_count=pk["cu"][B:B + 1])
    torch.cuda.synchronize()
    c.poll()
    n_tok = B + int(pk["cu"][B].item())
    t, cnt = c.table()
    assert cnt["observations"] == 3 and cnt["rebuilds"] == 3
    assert t[n_tok] != 7.0 and t[n_tok] > 0.0
    assert all(v == 7.0 for n, v in enumerate(t) if n != n_tok)
    c.close()


def test_poll_never_waits_for_a_running_step():
    c = sv.CostCurve(np.full(9, 1.0, np.float32), window=4, min_samples=1, rebuild_every=1)
    c.begin()
    torch.cuda._sleep(200_000_000)        # about 0.1 s of GPU spin at 2 GHz
    c.end(4)
    c.poll()
    _, cnt = c.table()
    assert cnt["pending"] == 1 and cnt["observations"] == 0
    torch.cuda.synchronize()
    c.poll()
    t, cnt = c.table()
    assert cnt["pending"] == 0 and cnt["observations"] == 1 and t[4] > 10.0
    c.close()


def test_upload_changes_what_the_pipeline_picks():
    B, kmax, V, H = 8, 5, 4096, 256
    inp = workloads.make_verify_inputs("batch64", 21, B=B, N=kmax, V=V)
    conf = workloads.make_confidence_inputs(21, B=B, kmax=kmax, H=H, n_max=64)
    t = lambda a, dt: torch.as_tensor(np.asarray(a, np.float32)).cuda().to(dt)  # noqa: E731
    dq = t(inp["draft_logits"], torch.bfloat16).view(B, kmax, V)
    dp = t(inp["target_logits"], torch.bfloat16).view(B, kmax + 1, V)
    x = torch.as_tensor(inp["draft_tokens"]).cuda().view(B, kmax)
    T = torch.ones(B, dtype=torch.float32, device="cuda")
    hidden, w = t(conf["hidden"], torch.bfloat16), t(conf["w"], torch.bfloat16)
    flat = np.full(65, 1.0, np.float32)               # every count costs the same: verify all
    vm = torch.as_tensor(flat).cuda()
    pl = sv.SpecPipeline(hidden, w, 4.0, vm, dq, dp, x, T, rule=1, seed=1, step=0)
    k0 = pl.launch()["k"].clone()
    steep = np.full(65, 1.0e6, np.float32)
    steep[:2] = 1.0                                   # only one-token passes are affordable
    c = sv.CostCurve(flat, window=4, min_samples=1, rebuild_every=4)
    for _ in range(4):
        c.observe(1, 1.0)
    for n in range(2, 65):
        for _ in range(4):
            c.observe(n, 1.0e6)
    assert np.array_equal(np.float32(c.table()[0]), steep)
    c.upload(vm)
    k1 = pl.launch()["k"].clone()
    torch.cuda.synchronize()
    assert np.array_equal(vm.cpu().numpy(), steep)
    assert (k0.cpu().numpy() == kmax).all(), k0
    assert (k1.cpu().numpy() == 0).all(), k1
    pl.close()
    c.close()


def test_begin_on_a_capturing_stream_is_refused():
    c = sv.CostCurve(np.full(9, 1.0, np.float32))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    a = torch.zeros(16, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        with pytest.raises(sv.SpecError) as e:
            c.begin()
        a += 1.0
    assert e.value.code == -1 and "capturing" in str(e.value)
    g.replay()
    torch.cuda.synchronize()
    assert a[0].item() == 1.0
    c.close()
