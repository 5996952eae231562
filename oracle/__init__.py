"""CPU oracle for the sequential-MTP hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 restatement of what the pages define:

* ``rows``   -- the semantic row compiler of "M7.6 - DeepSeek MTP" §0x04C,
                label ownership of "M7.4 - Multi-Token Prediction Foundations"
                §0x01A/§0x03A and the label counts of M7.6 §0x05A;
* ``chain``  -- the MTP module equations of M7.6 §0x03/§0x03C (dual RMSNorm,
                concat, 2d->d projection, one pre-norm block, shared head) run
                over the compiled rows as in the training loop of §0x06A, the
                per-depth loss of §0x05 and the vocabulary cross-entropy steps of
                M7.4 §0x06F;
* ``verify`` -- exact speculative selection: the one-proposal selector of
                M7.6 §0x09 generalised to γ drafts by the left-to-right rule of
                the speculative-decoding page, with Philox4x32-10 uniforms
                (Salmon et al., SC'11).

It shares no code with the CUDA path: no kernels, headers, helpers or tables.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import it; the product path never does.

Parity status: masks, RMSNorm, attention, CE/LSE, loss assembly and the
verifier are pinned by tests against the pages' worked numbers, closed forms,
invariants and brute force.  The whole-chain composition has no printed
numeric output on the pages: beyond its pinned components and the
packing/causality invariants it is "parity unpinned".
"""
