"""CPU oracle (test infrastructure): a plain fp64 restatement of Laplacian-kernel
Nystrom attention, used only by the tests, the smoke check and the benchmark's
CPU baseline."""
