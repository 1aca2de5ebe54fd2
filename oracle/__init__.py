"""CPU oracle for the Whisper transcription hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy restatement of what the hot path computes, used to
check the CUDA library.  Only the test suite, the smoke check and the CPU
baseline leg of the benchmark may import it; the library itself never does, and
this package imports nothing from the library.

Modules
  mel        audio -> 30 s chunks -> log-Mel spectrogram
  e4m3       OCP FP8 E4M3 encode / decode and the per-tensor scale rules
  model      conv stem, encoder, teacher-forced decoder, greedy argmax
  plan       chunk table and HBM wave packing (integer bookkeeping)

Sources (web pages on Whisper serving, cited by title and section):
  [BFW]  "Blazingly fast whisper transcriptions with Inference Endpoints"
         (Hugging Face blog) -- sections "Inference Stack", "Benchmarks".
  [TWT]  "TheStageAI/thewhisper-large-v3-turbo" model card -- "NVIDIA Usage",
         "Benchmarking Methodology".
  [WB]   "whisper-blaze 0.1.8" (PyPI page) -- "Batch Transcription",
         "VRAM usage guide", "Precision Presets", "GPU Mel Spectrogram",
         "Direct Kernel API".
  [UOW]  "Unlocking the power of OpenAI's Whisper" -- section 1 "The Whisper
         Architecture Deep Dive", 2 "Mel Spectrogram Generation and
         Optimization", 3 "Transformer Architecture in Whisper".

The pages fix the pipeline and its interfaces but print no constants; the
numeric hyper-parameters (n_fft 400, hop 160, mel counts, the log10 clamp, the
max-8 floor, the (x+4)/4 scaling, model widths) are those of the workloads this
oracle is checked on, and each reading taken where the pages are silent is
stated in the function that takes it.

Parity status: every function here is pinned by a CPU test against a closed
form, a brute-force definition, an independent library routine or an invariant
(tests/test_oracle_*.py); none is "parity unpinned".
"""
from . import e4m3, mel, model, plan  # noqa: F401
