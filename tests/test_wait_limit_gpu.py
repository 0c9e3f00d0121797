"""The bounded device waits: thread blocks meet at the grid barrier the
persistent kernels use (the fused Markov draft, the temperature-scaling fit),
once with every arrival made and once told to expect an arrival that never
comes.  The second wait must end by its time limit with a timeout status in
every block, and the device must stay usable.  Nothing else is in flight
while the blocks wait (no copy, MMA or tensor memory)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import verify_dspark_markov_gb300 as ds
    from verify_dspark_markov_gb300 import binding, build
    build.build()
    ds.load()
    return binding


def test_barrier_completes_when_every_block_arrives(ds):
    status, waited = ds.wait_selftest(blocks=8, missing=0, limit_us=500_000)
    torch.cuda.synchronize()
    assert status.tolist() == [ds.REQ_OK] * 8
    assert int(waited.max()) < 500_000_000


def test_wait_ends_by_its_limit_and_the_device_stays_usable(ds):
    limit_us = 50_000
    status, waited = ds.wait_selftest(blocks=4, missing=1, limit_us=limit_us)
    torch.cuda.synchronize()
    assert status.tolist() == [ds.REQ_TIMEOUT] * 4
    # the first block to give up waited the whole limit; the others stop on its error word
    assert int(waited.max()) >= limit_us * 1000
    assert int(waited.max()) < 2_000_000_000
    # the context is intact: a greedy verify runs and decides as expected
    g = torch.Generator(device="cpu").manual_seed(3)
    target = torch.randn((2, 3, 64), generator=g).to("cuda")
    proposals = target[:, :2, :].argmax(-1).to(torch.int32).contiguous()
    out_tokens, num_accepted, st = ds.verify(target, proposals)
    torch.cuda.synchronize()
    assert num_accepted.tolist() == [2, 2]
    assert st.tolist() == [ds.REQ_OK, ds.REQ_OK]
